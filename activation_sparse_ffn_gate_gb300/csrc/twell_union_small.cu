// twell_union_small.cu -- tensor-core kernels for small batches with the weights on the M side of
// the products: the union path's gate + up (and, gate only, the walk path's gate) for up to 128
// tokens, and the union path's down product for up to 512 tokens.
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
//      h = a * u (fp16; a = the packed value, 0 where g <= 0). The two CTAs of a cluster hold the
//      two halves of a 128-unit block: with T = 128 the second CTA's entries follow the first's,
//      whose per-token counts it reads from the first CTA's shared memory (distributed shared
//      memory). With T = 64 each CTA is a tile.
//      The K loop streams the CTA's 512 KB of Wg_s and Wu_s rows (d_model 2048) through a ring of
//      6-9 stages; at 64 tokens it runs at ~57 GB/s per SM (88 SMs: ~5 TB/s of HBM).
//   At 256 tokens this orientation was slower than the SM-pair tiles (45 against 40 us on the
//   1.5B-like layer: the N = 256 MMAs and 1 MB of x per CTA from L2), so it stops at 128.
//   2. down_small_kernel: y^T = Wd16t_s H^T, one 128-row block of Wd16t_s (128 columns of y) and
//      one tile of up to NP tokens per cluster of up to 8 CTAs, each a K range of f_pad; the fp32
//      partials meet in the cluster's shared memory and are added in rank order (a fixed order)
//      into bf16 y. It also serves the union path's down product for 129-512 tokens (128-token
//      tiles), after the SM-pair gate + up GEMM.
// Both launch as programmatic dependents of the kernel before them on the stream.
#include <cooperative_groups.h>

#include <algorithm>

#include "twell_gemm.cuh"

namespace twell {
namespace {

constexpr int kSmallUnits = 64;        // hidden units per CTA
constexpr int kSmallThreads = 192;     // warp 0 TMA, warp 1 TMEM + MMA, warps 2..5 epilogue
// gate + up: the same roles, two more warps; after the main loop all eight pack (one token and
// 32-unit half per thread for up to 128 tokens)
constexpr int kGateUpThreads = 256;
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

// GATE_ONLY (the walk path's gate): the A tile's first 64 rows are the units' Wg_s rows and the
// rest is not loaded (its products, in TMEM lanes 64-127, are never read); the epilogue packs the
// TwELL only.
template <int NP, bool GATE_ONLY>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGateUpThreads, 1)
    gate_up_small_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmU,
                         const __grid_constant__ CUtensorMap tmX, const SmallArgs a)
{
    using C = SmallCfg<NP>;
    constexpr int STAGES = C::STAGES;
    constexpr uint32_t IDESC = idesc_bf16_f32(128, NP, false, false);
    constexpr uint32_t LOAD_BYTES = GATE_ONLY ? C::A_BYTES / 2 + C::B_BYTES : C::STAGE_BYTES;
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
    // only now may the down kernel start: it reads Wd16t_s before its own wait, so every kernel
    // before this call must have completed by then
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    bool have_acc = false;
    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
            for (int kb = 0; kb < kbs; ++kb) {
                if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status, a.wait_limit_ns)) break;
                uint8_t* sa = smem + stage * C::STAGE_BYTES;
                const int k0 = kb * kBK;
                mbar_arrive_expect_tx(&full[stage], LOAD_BYTES);
                tma_load_2d(sa, &tmG, k0, u0, &full[stage]);
                if constexpr (!GATE_ONLY) tma_load_2d(sa + 8192, &tmU, k0, u0, &full[stage]);
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
    } else if (warp < 6) {
        // ------------------------------------------------------------------ TMEM -> shared memory
        const int q = warp & 3;  // TMEM lanes 32q .. 32q + 31: rows 0-63 hold g, 64-127 u
        int ok = 1;
        if (lane == 0) ok = wait_bounded(tfull, 0, abort_flag, a.status, a.wait_limit_ns) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && !(GATE_ONLY && q >= 2)) {
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
    // Pack thread (all eight warps): one 32-unit half hf of this CTA's units for token tb (< N).
    const bool wide = a.T == 128;
    const bool second = wide && rank == 1;
    const int tile = wide ? blockIdx.x / 2 : blockIdx.x;
    const int hf = warp & 1, tb = 32 * (warp >> 1) + lane;
    constexpr int TSTEP = kGateUpThreads / 2;  // tokens per pass of all threads (N <= 128: one pass)
    const int uh = u0 + 32 * hf;  // global index of the half's first unit
    const int nin = min(max(a.f - uh, 0), 32);  // its units below f
    // 1. counts of kept units per token and half
    if (have) {
        for (int t = tb; t < a.N; t += TSTEP) {
            int c = 0;
#pragma unroll 8
            for (int j = 0; j < 32; ++j) c += (j < nin && gs[(32 * hf + j) * GP + t] > 0.0f) ? 1 : 0;
            ch_s[hf * NP + t] = c;
        }
    }
    if (have) bar_or(1, kGateUpThreads, false);  // ch_s is complete
    if (wide && !second && have && hf == 0)
        for (int t = tb; t < a.N; t += TSTEP) cnt_s[t] = ch_s[t] + ch_s[NP + t];

    // 2. per token and half: ReLU + TwELL in ascending unit order, as twell_gate_pack packs, and
    // h = a * u (a = the value as packed) as fp16, 16 bytes at a time
    auto pack = [&]() {
        const int ioff = (second ? kSmallUnits : 0) + 32 * hf;  // index within the tile of unit j = 0
        __nv_bfloat16* vals16 = static_cast<__nv_bfloat16*>(a.vals);
        float* vals32 = static_cast<float*>(a.vals);
        bool over = false;
        for (int t = tb; t < a.N; t += TSTEP) {
            const int base = (second ? base_s[t] : 0) + (hf ? ch_s[t] : 0);
            const size_t slot = (static_cast<size_t>(t) * a.nt + tile) * static_cast<size_t>(a.T) + base;
            float gr[32], ur[32];  // all loads first: the stores below may not be moved above them
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                gr[j] = gs[(32 * hf + j) * GP + t];
                ur[j] = GATE_ONLY ? 0.0f : us[(32 * hf + j) * GP + t];
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
                if (!GATE_ONLY && uh + j0 < a.ldo)  // ldo is a multiple of 64: the half is whole
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
    if (!second && have) pack();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (second) {
        have = have && !*cluster.map_shared_rank(const_cast<int*>(abort_flag), 0);
        if (have) {
            const int* peer_cnt = cluster.map_shared_rank(cnt_s, 0);
            for (int t = static_cast<int>(threadIdx.x); t < a.N; t += kGateUpThreads) base_s[t] = peer_cnt[t];
            bar_or(1, kGateUpThreads, false);  // base_s is complete (its loads have returned)
        }
    }
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (second && have) pack();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Down product of the small-batch path: y^T = Wd16t_s H^T for one 128-row block of Wd16t_s (128
// output columns of y) per cluster of ks CTAs, CTA r taking the r-th of ks near-equal K ranges of
// f_pad (fp16 operands, A = Wd16t_s rows K-major, B = H [NP, 64] per k-block, one tcgen05.mma of
// M = 128, N = NP per 16 of K). Its fp32 partial goes from TMEM to shared memory as [token][row];
// after a cluster barrier CTA r adds, for its ~128 / ks rows, the ks partials in rank order (a
// fixed order) from the cluster's shared memory, 16 bytes at a time, and writes those columns of y
// in bf16.
struct DownArgs {
    int N, d, fp, ks;
    int m_tiles;  // 128-row blocks of Wd16t_s; cluster c takes block c % m_tiles of token tile c / m_tiles
    __nv_bfloat16* y;
    int32_t* status;
    uint64_t wait_limit_ns;
};

constexpr int kDownMaxCluster = 8;

template <int NP>
struct DownCfg {
    static constexpr uint32_t A_BYTES = 128 * kBK * 2;
    static constexpr uint32_t B_BYTES = NP * kBK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = kSmallRing / STAGE_BYTES < 10 ? static_cast<int>(kSmallRing / STAGE_BYTES) : 10;
    static constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 256;
    static_assert(128u * NP * 4 <= STAGES * STAGE_BYTES, "the partial fits in the ring it replaces");
};

template <int NP>
__global__ void __launch_bounds__(kSmallThreads, 1)
    down_small_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                      const DownArgs a)
{
    using C = DownCfg<NP>;
    constexpr int STAGES = C::STAGES;
    constexpr uint32_t IDESC = idesc_f16_f32(128, NP, false, false);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* drain = tfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* P = reinterpret_cast<float*>(smem);  // after the main loop: the partial [token][128 rows]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    const int ks = a.ks;
    const int r = static_cast<int>(cluster.block_rank());
    const int blk = static_cast<int>(blockIdx.x) / ks;
    const int m0 = blk % a.m_tiles * 128, t0 = blk / a.m_tiles * NP;  // rows of Wd16t_s, first token
    const int nt_here = min(NP, a.N - t0);
    const int kbs = a.fp / kBK;
    const int kb0 = kbs * r / ks, kb1 = kbs * (r + 1) / ks;  // non-empty: ks <= kbs

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
    // The first stages' Wd16t_s tiles are requested before the wait for the previous grid: no
    // kernel that can still be running writes Wd16t_s (the kernel before this one on the stream
    // lets it start only after its own wait, or started after all earlier work had completed).
    const int npre = min(kb1 - kb0, STAGES);
    if (threadIdx.x == 0) {  // the thread that initialised the barriers
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmH);
        for (int i = 0; i < npre; ++i) {
            mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
            tma_load_2d(smem + i * C::STAGE_BYTES, &tmW, (kb0 + i) * kBK, m0, &full[i]);
        }
    }
    if (warp == 1) {
        tmem_alloc<1>(tmem_slot, NP);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // H is the previous grid's output

    bool have_acc = false;
    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                uint8_t* sa = smem + stage * C::STAGE_BYTES;
                if (kb - kb0 >= npre) {  // (the first npre stages are free and hold their A tile already)
                    if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status, a.wait_limit_ns)) break;
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    tma_load_2d(sa, &tmW, kb * kBK, m0, &full[stage]);
                }
                tma_load_2d(sa + C::A_BYTES, &tmH, kb * kBK, t0, &full[stage]);
                issued_mask |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if (issued_mask & (1u << s))
                    wait_bounded(&full[s], (issued_phase >> s) & 1u, nullptr, a.status, a.wait_limit_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
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
                                  (kb != kb0 || k != 0) ? 1u : 0u);
                tc_commit<1>(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) tc_commit<1>(tfull);
            tc_commit<1>(drain);
            wait_bounded(drain, 0, nullptr, a.status, a.wait_limit_ns);
        }
    } else {
        const int q = warp & 3;
        int ok = 1;
        if (lane == 0) ok = wait_bounded(tfull, 0, abort_flag, a.status, a.wait_limit_ns) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
            tc_fence_after();
            float* dst = P + 32 * q + lane;
#pragma unroll 1
            for (int ch = 0; ch < NP / 32; ++ch) {
                float v[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + ch * 32, v);
#pragma unroll
                for (int k = 0; k < 32; ++k) dst[(ch * 32 + k) * 128] = v[k];
            }
            have_acc = true;
        }
    }
    tc_fence_before();
    int have = __syncthreads_or(have_acc ? 1 : 0) && !*abort_flag;
    tc_fence_after();
    if (warp == 1) tmem_dealloc<1>(tmem_base, NP);
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");  // every partial is in place
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    const float* part[kDownMaxCluster];
#pragma unroll
    for (int i = 0; i < kDownMaxCluster; ++i) {
        part[i] = cluster.map_shared_rank(P, i < ks ? i : 0);
        if (i < ks) have = have && !*cluster.map_shared_rank(const_cast<int*>(abort_flag), i);
    }
    if (have) {
        // rows [j0, j1) of the block (multiples of 4), four at a time: element e = token e / n4, rows
        // j0 + 4 (e % n4) .. + 3; consecutive threads read 16 consecutive bytes of each partial
        const int j0 = 128 * r / ks / 4 * 4, j1 = r + 1 == ks ? 128 : 128 * (r + 1) / ks / 4 * 4;
        const int n4 = (j1 - j0) / 4, total = n4 * nt_here;
        for (int e0 = threadIdx.x; e0 < total; e0 += 2 * kSmallThreads) {
            float4 v[2][kDownMaxCluster];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int e = min(e0 + b * kSmallThreads, total - 1);
                const int off = (e / n4) * 128 + j0 + 4 * (e % n4);
#pragma unroll
                for (int i = 0; i < kDownMaxCluster; ++i)
                    v[b][i] = i < ks ? *reinterpret_cast<const float4*>(part[i] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int e = e0 + b * kSmallThreads;
                if (e >= total) break;
                float4 acc = v[b][0];
#pragma unroll
                for (int i = 1; i < kDownMaxCluster; ++i)
                    if (i < ks) {
                        acc.x += v[b][i].x;
                        acc.y += v[b][i].y;
                        acc.z += v[b][i].z;
                        acc.w += v[b][i].w;
                    }
                const int col = m0 + j0 + 4 * (e % n4);
                __nv_bfloat16* o = a.y + static_cast<size_t>(t0 + e / n4) * a.d + col;
                if (col + 3 < a.d) {  // d is a multiple of 8: y rows are 16-byte aligned, col a multiple of 4
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
                    uint2 w;
                    w.x = *reinterpret_cast<const uint32_t*>(&lo);
                    w.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(o) = w;
                } else {
                    const float av[4] = {acc.x, acc.y, acc.z, acc.w};
                    for (int k = 0; k < 4 && col + k < a.d; ++k) o[k] = __float2bfloat16_rn(av[k]);
                }
            }
        }
    }
    // the partials stay in place until every CTA of the cluster has read them (relaxed: this
    // barrier orders no memory, so no thread waits here for its stores to drain)
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <int NP, bool GATE_ONLY>
twell_status launch_gate_up_small(const void* x, const void* Wg_s, const void* Wu_s, const SmallArgs& a,
                                  cudaStream_t s)
{
    using C = SmallCfg<NP>;
    CUtensorMap tg, tu, tx;
    twell_status st = twell_host::make_tmap_bf16(&tg, Wg_s, a.d, a.f, a.d, 64, kSmallUnits);
    if (st != TWELL_OK) return st;
    tu = tg;
    if (!GATE_ONLY) st = twell_host::make_tmap_bf16(&tu, Wu_s, a.d, a.f, a.d, 64, kSmallUnits);
    if (st != TWELL_OK) return st;
    st = twell_host::make_tmap_bf16(&tx, x, a.d, a.N, a.d, 64, NP);
    if (st != TWELL_OK) return st;
    auto kern = gate_up_small_kernel<NP, GATE_ONLY>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM_BYTES)) !=
        cudaSuccess)
        return TWELL_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * static_cast<unsigned>((a.f + 127) / 128));
    cfg.blockDim = dim3(kGateUpThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tg, tu, tx, a) != cudaSuccess) return TWELL_ERR_CUDA;
    return twell_host::launch_status();
}

template <int NP>
twell_status launch_down_small(const __half* H, const void* Wd16t_s, int N, int d, int f, int fp, void* y,
                               int32_t* dev_status, cudaStream_t s)
{
    using C = DownCfg<NP>;
    twell_host::DevInfo di;
    if (twell_host::dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    const int m_tiles = (d + 127) / 128;
    const int blocks = m_tiles * ((N + NP - 1) / NP);  // (row block, token tile) pairs
    auto kern = down_small_kernel<NP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM_BYTES)) !=
        cudaSuccess)
        return TWELL_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kSmallThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // K ranges per block: the largest cluster (up to 8) of which all blocks fit on the GPU at once
    // (clusters are placed within one GPC: fewer of 8 fit than SMs / 8); counts cached per size
    static int fit[kDownMaxCluster + 1][3] = {};
    const int slot = NP == 32 ? 0 : (NP == 64 ? 1 : 2);
    int ks = 1;
    for (int c = std::min(kDownMaxCluster, fp / kBK); c > 1; --c) {
        if (fit[c][slot] == 0) {
            attr[0].val.clusterDim.x = static_cast<unsigned>(c);
            cfg.gridDim = dim3(static_cast<unsigned>(c * blocks));
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return TWELL_ERR_CUDA;
            fit[c][slot] = n > 0 ? n : -1;
        }
        if (fit[c][slot] >= blocks) {
            ks = c;
            break;
        }
    }
    CUtensorMap tw, th;
    twell_status st = twell_host::make_tmap_bf16(&tw, Wd16t_s, f, d, f, 64, 128);
    if (st != TWELL_OK) return st;
    st = twell_host::make_tmap_bf16(&th, H, fp, N, fp, 64, NP);
    if (st != TWELL_OK) return st;
    DownArgs a{N, d, fp, ks, m_tiles, static_cast<__nv_bfloat16*>(y), dev_status, twell_host::wait_limit_ns()};
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks * ks));
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, tw, th, a) != cudaSuccess) return TWELL_ERR_CUDA;
    return twell_host::launch_status();
}

}  // namespace
}  // namespace twell

twell_status twell_host::gate_up_small(const void* x, const void* Wg_s, const void* Wu_s, int N, int d, int f, int T,
                                       const twell_packed* out, __half* H, int ldo, int32_t* dev_status,
                                       cudaStream_t s)
{
    if (N <= 0 || N > kTransposedMaxN || (T != 64 && T != 128)) return TWELL_ERR_UNSUPPORTED;
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
    if (Wu_s == nullptr) {
        if (N <= 32) return twell::launch_gate_up_small<32, true>(x, Wg_s, Wu_s, a, s);
        if (N <= 64) return twell::launch_gate_up_small<64, true>(x, Wg_s, Wu_s, a, s);
        return twell::launch_gate_up_small<128, true>(x, Wg_s, Wu_s, a, s);
    }
    if (N <= 32) return twell::launch_gate_up_small<32, false>(x, Wg_s, Wu_s, a, s);
    if (N <= 64) return twell::launch_gate_up_small<64, false>(x, Wg_s, Wu_s, a, s);
    return twell::launch_gate_up_small<128, false>(x, Wg_s, Wu_s, a, s);
}

twell_status twell_host::down_small(const __half* H, const void* Wd16t_s, int N, int d, int f, int fp, void* y,
                                    int32_t* dev_status, cudaStream_t s)
{
    if (N <= 0 || N > kDownSmallMaxN || fp % 64 != 0) return TWELL_ERR_UNSUPPORTED;
    if (N <= 32) return twell::launch_down_small<32>(H, Wd16t_s, N, d, f, fp, y, dev_status, s);
    if (N <= 64) return twell::launch_down_small<64>(H, Wd16t_s, N, d, f, fp, y, dev_status, s);
    return twell::launch_down_small<128>(H, Wd16t_s, N, d, f, fp, y, dev_status, s);  // 128-token tiles
}
