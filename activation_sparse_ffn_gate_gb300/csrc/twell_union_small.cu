// twell_union_small.cu -- the union path for batches of at most 128 tokens, with the weights on the
// M side of the tensor-core products.
//
// For a batch of N <= 128 tokens the union path's 256 x 256 SM-pair tiles put the tokens on the
// 256-row side: at 64 tokens 75% of every MMA is padding rows, and each tile's tensor work outlasts
// the streaming of its weight rows. Here the products run transposed, so that the MMA's M = 128
// side holds weight rows and the tokens are its N = NP columns (NP = N rounded up to 32, 64 or 128):
//
//   1. gate_up_small_kernel: CTA c holds 64 hidden units; its A tile stacks their 64 rows of Wg_s
//      over their 64 rows of Wu_s (two TMA boxes into one 128-row, 128-byte-swizzled tile), B is x
//      [NP, 64] per k-block, and one tcgen05.mma (cta_group::1, M = 128, N = NP) per 16 of K
//      accumulates [g; u]^T of the 64 units for all tokens into TMEM. The epilogue moves g and u
//      to shared memory as [unit][token]; one thread per token and 32-unit half counts, then
//      packs its units exactly as twell_gate_pack packs (ReLU, ascending unit order), storing
//      h = a * u (fp16; a = the packed value, 0 where g <= 0). The two CTAs of a cluster hold the two halves of a 128-unit block: with T = 128
//      the second CTA's entries follow the first's, whose per-token counts it reads from the
//      first CTA's shared memory (distributed shared memory). With T = 64 each CTA is a tile.
//   2. the down product y^T = Wd16t_s H^T on the generic tcgen05 GEMM (A = Wd16t_s [d, f] fp16,
//      B = H [N, f_pad] fp16, both K-major, a 128 x NP tile), split along K into ks ranges so that
//      ceil(d / 128) * ks work units fill the SMs; fp32 partials [ks][d][NP];
//   3. reduce_splits_t_bf16_kernel adds the partials in range order (a fixed order) and writes
//      y [N, d] in bf16 through a 32 x 32 shared-memory transpose.
// All three launch as programmatic dependents of the kernel before them on the stream.
#include <cooperative_groups.h>

#include <algorithm>

#include "twell_gemm.cuh"

namespace twell {
namespace {

constexpr int kSmallUnits = 64;        // hidden units per CTA
constexpr int kSmallThreads = 192;     // warp 0 TMA, warp 1 TMEM + MMA, warps 2..5 epilogue
constexpr uint32_t kSmallRing = 196608;  // shared memory of the operand ring (and, after it, of g and u)

template <int NP>
struct SmallCfg {
    static constexpr uint32_t A_BYTES = 128 * kBK * 2;  // 64 rows of Wg_s over 64 rows of Wu_s
    static constexpr uint32_t B_BYTES = NP * kBK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = kSmallRing / STAGE_BYTES < 10 ? static_cast<int>(kSmallRing / STAGE_BYTES) : 10;
    // g and u as [unit][NP + 1] fp32, then four counts per token
    static constexpr uint32_t GU_BYTES = 2u * kSmallUnits * (NP + 1) * 4 + 4u * NP * 4;
    static constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 256;
    static_assert(GU_BYTES <= STAGES * STAGE_BYTES, "g, u and the counts fit in the ring they replace");
    static_assert(B_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
};

struct SmallArgs {
    int N, d, f, T, nt, ldo;  // ldo: row pitch of H (f rounded up to 64)
    int vals_f32;
    void* vals;
    uint8_t* idx;
    uint16_t* cnt;
    __half* H;
    int32_t* status;
    uint64_t wait_limit_ns;
};

template <int NP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kSmallThreads, 1)
    gate_up_small_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmU,
                         const __grid_constant__ CUtensorMap tmX, const SmallArgs a)
{
    using C = SmallCfg<NP>;
    constexpr int STAGES = C::STAGES;
    constexpr uint32_t IDESC = idesc_bf16_f32(128, NP, false, false);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* drain = tfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // after the main loop, over the ring: g and u as [unit][token] (row pitch NP + 1, so that both
    // the per-unit writes and the per-token reads are free of bank conflicts), then per token the
    // counts of the two 32-unit halves and, for a 128-wide tile, the first CTA's total
    constexpr int GP = NP + 1;
    float* gs = reinterpret_cast<float*>(smem);
    float* us = gs + kSmallUnits * GP;
    int* ch_s = reinterpret_cast<int*>(us + kSmallUnits * GP);  // [2][NP]
    int* cnt_s = ch_s + 2 * NP;                                   // first CTA: its count per token
    int* base_s = cnt_s + NP;                                     // second CTA: the same, copied

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int u0 = blockIdx.x * kSmallUnits;
    const int kbs = (a.d + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmG);
        tma_prefetch_desc(&tmU);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc<1>(tmem_slot, NP);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // x and the weights are the previous grids' to write

    bool have_acc = false;
    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
            for (int kb = 0; kb < kbs; ++kb) {
                if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status, a.wait_limit_ns)) break;
                uint8_t* sa = smem + stage * C::STAGE_BYTES;
                const int k0 = kb * kBK;
                mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                tma_load_2d(sa, &tmG, k0, u0, &full[stage]);
                tma_load_2d(sa + 8192, &tmU, k0, u0, &full[stage]);
                tma_load_2d(sa + C::A_BYTES, &tmX, k0, 0, &full[stage]);
                issued_mask |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // every copy issued has landed before the ring is reused or the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if (issued_mask & (1u << s))
                    wait_bounded(&full[s], (issued_phase >> s) & 1u, nullptr, a.status, a.wait_limit_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int kb = 0; kb < kbs; ++kb) {
                if (!wait_bounded(&full[stage], phase, abort_flag, a.status, a.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                    tc_mma_f16<1>(tmem_base, desc_sw128(a_addr + k * 32, 16), desc_sw128(b_addr + k * 32, 16), IDESC,
                                  (kb != 0 || k != 0) ? 1u : 0u);
                tc_commit<1>(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) tc_commit<1>(tfull);
            // every tcgen05 operation issued has completed before TMEM is read back or freed
            tc_commit<1>(drain);
            wait_bounded(drain, 0, nullptr, a.status, a.wait_limit_ns);
        }
    } else {
        // ------------------------------------------------------------------ TMEM -> shared memory
        const int q = warp & 3;  // TMEM lanes 32q .. 32q + 31: rows 0-63 hold g, 64-127 u
        int ok = 1;
        if (lane == 0) ok = wait_bounded(tfull, 0, abort_flag, a.status, a.wait_limit_ns) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
            tc_fence_after();
            const int row = 32 * q + lane;
            float* dst = (row < kSmallUnits ? gs : us) + (row % kSmallUnits) * GP;
#pragma unroll 1
            for (int ch = 0; ch < NP / 32; ++ch) {
                float v[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + ch * 32, v);
#pragma unroll
                for (int k = 0; k < 32; ++k) dst[ch * 32 + k] = v[k];
            }
            have_acc = true;
        }
    }
    // g and u are in shared memory, unless a wait gave up (TWELL_ERR_TIMEOUT is reported): then
    // this CTA packs nothing
    tc_fence_before();
    int have = __syncthreads_or(have_acc ? 1 : 0) && !*abort_flag;
    tc_fence_after();
    if (warp == 1) tmem_dealloc<1>(tmem_base, NP);
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    // T = 128: the cluster's two CTAs hold units [0, 64) and [64, 128) of tile blockIdx.x / 2; each
    // packs its own units, the second CTA's entries after the first's (its per-token counts, read
    // once from the first CTA's shared memory). T = 64: each CTA is a tile of its own.
    // Epilogue thread: one 32-unit half hf of this CTA's units for tokens tb, tb + 64 (< N).
    const bool wide = a.T == 128;
    const bool second = wide && rank == 1;
    const int tile = wide ? blockIdx.x / 2 : blockIdx.x;
    const int ew = warp - 2, hf = ew & 1, tb = 32 * (ew >> 1) + lane;
    const int uh = u0 + 32 * hf;  // global index of the half's first unit
    const int nin = min(max(a.f - uh, 0), 32);  // its units below f
    // 1. counts of kept units per token and half
    if (have && warp >= 2) {
        for (int t = tb; t < a.N; t += 64) {
            int c = 0;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) c += (j < nin && gs[(32 * hf + j) * GP + t] > 0.0f) ? 1 : 0;
            ch_s[hf * NP + t] = c;
        }
    }
    if (have && warp >= 2) bar_or(1, 128, false);  // the four epilogue warps: ch_s is complete
    if (wide && !second && have && warp >= 2 && hf == 0)
        for (int t = tb; t < a.N; t += 64) cnt_s[t] = ch_s[t] + ch_s[NP + t];

    // 2. per token and half: ReLU + TwELL in ascending unit order, as twell_gate_pack packs, and
    // h = a * u (a = the value as packed) as fp16, 16 bytes at a time
    auto pack = [&]() {
        const int ioff = (second ? kSmallUnits : 0) + 32 * hf;  // index within the tile of unit j = 0
        __nv_bfloat16* vals16 = static_cast<__nv_bfloat16*>(a.vals);
        float* vals32 = static_cast<float*>(a.vals);
        bool over = false;
        for (int t = tb; t < a.N; t += 64) {
            const int base = (second ? base_s[t] : 0) + (hf ? ch_s[t] : 0);
            const size_t slot = (static_cast<size_t>(t) * a.nt + tile) * static_cast<size_t>(a.T) + base;
            float gr[32], ur[32];  // all loads first: the stores below may not be moved above them
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                gr[j] = gs[(32 * hf + j) * GP + t];
                ur[j] = us[(32 * hf + j) * GP + t];
            }
            int c = 0;
#pragma unroll
            for (int j0 = 0; j0 < 32; j0 += 8) {
                uint32_t hw[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float hv[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int j = j0 + e + k;
                        const float gv = gr[j];
                        const bool keep = j < nin && gv > 0.0f;
                        const float av = a.vals_f32 ? gv : __bfloat162float(__float2bfloat16_rn(gv));
                        if (keep) {
                            if (a.vals_f32) vals32[slot + c] = av;
                            else vals16[slot + c] = __float2bfloat16_rn(av);
                            a.idx[slot + c] = static_cast<uint8_t>(ioff + j);
                            ++c;
                        }
                        hv[k] = keep ? av * ur[j] : 0.0f;
                        over |= !(fabsf(hv[k]) < 65520.0f);
                    }
                    const __half2 hh = __floats2half2_rn(hv[0], hv[1]);
                    hw[e / 2] = *reinterpret_cast<const uint32_t*>(&hh);
                }
                if (uh + j0 < a.ldo)  // ldo is a multiple of 64: the half is whole
                    *reinterpret_cast<uint4*>(a.H + static_cast<size_t>(t) * a.ldo + uh + j0) =
                        make_uint4(hw[0], hw[1], hw[2], hw[3]);
            }
            if (hf == 1 && tile < a.nt && (!wide || second))
                a.cnt[static_cast<size_t>(t) * a.nt + tile] = static_cast<uint16_t>(base + c);
        }
        if (over) report(a.status, TWELL_ERR_DEVICE_CHECK);
    };

    // Cluster barrier 1: the first CTA's counts are in place. Barrier 2 (relaxed: it orders no
    // memory, so no thread waits there for its stores to drain): the second CTA has read them,
    // so the first may exit.
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    if (!second && have && warp >= 2) pack();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (second) {
        have = have && !*cluster.map_shared_rank(const_cast<int*>(abort_flag), 0);
        if (have && warp >= 2) {
            const int* peer_cnt = cluster.map_shared_rank(cnt_s, 0);
            for (int t = static_cast<int>(threadIdx.x) - 64; t < a.N; t += 128) base_s[t] = peer_cnt[t];
            bar_or(1, 128, false);  // base_s is complete (its loads have returned)
        }
    }
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (second && have && warp >= 2) pack();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// y[t, j] = bf16(part[0][j][t] + ... + part[ks - 1][j][t]) (ks <= kMaxSplits) through a 32 x 32
// transpose in shared memory; every thread issues its ks loads before it adds them in order.
// Block (32, 32); grid (ceil(N / 32), ceil(d / 32)).
constexpr int kMaxSplits = 16;
__global__ void __launch_bounds__(1024) reduce_splits_t_bf16_kernel(const float* __restrict__ part, int ks,
                                                                    size_t split_stride, int ldp, int N, int d,
                                                                    __nv_bfloat16* __restrict__ y)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float tile[32][33];
    const int t0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    {
        const int j = j0 + ty, t = t0 + tx;
        const bool ok = j < d && t < N;
        const float* p = part + static_cast<size_t>(ok ? j : 0) * ldp + (ok ? t : 0);
        float v[kMaxSplits];
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) v[s] = (ok && s < ks) ? p[static_cast<size_t>(s) * split_stride] : 0.0f;
        float acc = v[0];
#pragma unroll
        for (int s = 1; s < kMaxSplits; ++s)
            if (s < ks) acc += v[s];
        tile[ty][tx] = acc;
    }
    __syncthreads();
    const int t = t0 + ty, j = j0 + tx;
    if (t < N && j < d) y[static_cast<size_t>(t) * d + j] = __float2bfloat16_rn(tile[tx][ty]);
}

template <int NP>
twell_status launch_gate_up_small(const void* x, const void* Wg_s, const void* Wu_s, const SmallArgs& a,
                                  cudaStream_t s)
{
    using C = SmallCfg<NP>;
    CUtensorMap tg, tu, tx;
    twell_status st = twell_host::make_tmap_bf16(&tg, Wg_s, a.d, a.f, a.d, 64, kSmallUnits);
    if (st != TWELL_OK) return st;
    st = twell_host::make_tmap_bf16(&tu, Wu_s, a.d, a.f, a.d, 64, kSmallUnits);
    if (st != TWELL_OK) return st;
    st = twell_host::make_tmap_bf16(&tx, x, a.d, a.N, a.d, 64, NP);
    if (st != TWELL_OK) return st;
    auto kern = gate_up_small_kernel<NP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM_BYTES)) !=
        cudaSuccess)
        return TWELL_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * static_cast<unsigned>((a.f + 127) / 128));
    cfg.blockDim = dim3(kSmallThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tg, tu, tx, a) != cudaSuccess) return TWELL_ERR_CUDA;
    return twell_host::launch_status();
}

// K ranges of the transposed down product: ceil(d / 128) * ks units fill the SMs at most once,
// each range four k-blocks or more, ks <= kSmallMaxSplits.
int small_down_splits(int d, int fp)
{
    twell_host::DevInfo di;
    if (twell_host::dev_info(&di) != TWELL_OK) return 1;
    const int m_tiles = (d + kBM - 1) / kBM;
    int ks = std::max(di.sm_count / m_tiles, 1);
    ks = std::min(ks, std::min(twell_host::kSmallMaxSplits, kMaxSplits));
    ks = std::min(ks, std::max(fp / kBK / 4, 1));
    return ks;
}

template <int NP>
twell_status launch_down_small(const __half* H, const void* Wd16t_s, int N, int d, int f, int fp, void* y, float* part,
                               int32_t* dev_status, cudaStream_t s)
{
    const int ks = small_down_splits(d, fp);
    GemmArgs g{};
    g.M = d;
    g.N = N;
    g.K = fp;
    g.k_splits = ks;
    g.split_stride = static_cast<int64_t>(d) * NP;
    g.out = part;
    g.ldo = NP;
    g.status = dev_status;
    g.pdl = 1;
    const twell_host::GemmOperand A{Wd16t_s, d, f, f}, B{H, N, fp, fp};
    twell_status st = twell_host::launch_gemm<NP, false, false, Epi::StoreF32, false, true>(A, B, nullptr, g, s);
    if (st != TWELL_OK) return st;
    return twell_host::launch_dep(reduce_splits_t_bf16_kernel, dim3((N + 31) / 32, (d + 31) / 32), dim3(32, 32), 0, s,
                                  static_cast<const float*>(part), ks, static_cast<size_t>(d) * NP, NP, N, d,
                                  static_cast<__nv_bfloat16*>(y)) == TWELL_OK
               ? twell_host::launch_status()
               : TWELL_ERR_CUDA;
}

}  // namespace
}  // namespace twell

twell_status twell_host::gate_up_small(const void* x, const void* Wg_s, const void* Wu_s, int N, int d, int f, int T,
                                       const twell_packed* out, __half* H, int ldo, int32_t* dev_status,
                                       cudaStream_t s)
{
    if (N <= 0 || N > kSmallMaxN || (T != 64 && T != 128)) return TWELL_ERR_UNSUPPORTED;
    twell::SmallArgs a{};
    a.N = N;
    a.d = d;
    a.f = f;
    a.T = T;
    a.nt = (f + T - 1) / T;
    a.ldo = ldo;
    a.vals_f32 = out->dtype == TWELL_F32 ? 1 : 0;
    a.vals = out->vals;
    a.idx = out->idx;
    a.cnt = out->cnt;
    a.H = H;
    a.status = dev_status;
    a.wait_limit_ns = wait_limit_ns();
    if (N <= 32) return twell::launch_gate_up_small<32>(x, Wg_s, Wu_s, a, s);
    if (N <= 64) return twell::launch_gate_up_small<64>(x, Wg_s, Wu_s, a, s);
    return twell::launch_gate_up_small<128>(x, Wg_s, Wu_s, a, s);
}

twell_status twell_host::down_small(const __half* H, const void* Wd16t_s, int N, int d, int f, int fp, void* y,
                                    float* part, int32_t* dev_status, cudaStream_t s)
{
    if (N <= 0 || N > kSmallMaxN) return TWELL_ERR_UNSUPPORTED;
    if (N <= 32) return twell::launch_down_small<32>(H, Wd16t_s, N, d, f, fp, y, part, dev_status, s);
    if (N <= 64) return twell::launch_down_small<64>(H, Wd16t_s, N, d, f, fp, y, part, dev_status, s);
    return twell::launch_down_small<128>(H, Wd16t_s, N, d, f, fp, y, part, dev_status, s);
}
