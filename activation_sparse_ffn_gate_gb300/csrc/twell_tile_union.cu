// twell_tile_union.cu -- the up and down projections of a TwELL layer as tensor-core GEMMs over
// the units each tile of 128 tokens keeps ("tile union"), with gathered weight rows.
//
// The pages' fused kernel gathers, for every token, the rows of Wu and Wd its kept units need
// ([TG] "Инференс"), and the heavy work belongs on the tensor cores ([TC] §3). On GB300 the two
// meet per tile of 128 tokens: the units any token of the tile keeps -- the tile's union U_m,
// 1 - (1 - p)^128 of d_ff at density p (43% on the 1.5B-like layer, 72% at 1%, 92% at 2%) -- are
// gathered as the B operand of a tcgen05 GEMM, so each weight row is read once per tile instead of
// once per token that keeps it, and the products run at tensor-core rate. Steps (one stream):
//   1. union_bits_kernel (warp per token row): the bits of the row's kept units in its tile's bitmap;
//      union_prefix_kernel (CTA per tile): U_m ascending (the rank of a unit in the bitmap is its
//      union position) and |U_m|; union_work_kernel: the up GEMM's blocks, 256 union positions each;
//   2. tile_expand_kernel (warp per row): H[r, p] = a (fp16) at the row's kept union positions and the
//      row's keep mask over positions (H itself is not cleared);
//   3. up GEMM: h = a * (x_m . Wu_s[U_m[p]]) in place in H, zeros where the mask bit is clear;
//      tcgen05 128 x 256 tiles, A = the x tile by TMA, B = 256 gathered rows of Wu_s (K-major);
//   4. down GEMM: y_m = H_m . Wd16_s[U_m] over K = |U_m|, A = the H tile by TMA, B = 64 gathered
//      rows of an fp16 copy of Wd_s per k-block (MN-major), y stored as bf16.
// The dense hidden activation exists only over each tile's union, in the workspace. h is rounded
// once to fp16 (11 significant bits); an h or a beyond the fp16 range is recorded as
// TWELL_ERR_DEVICE_CHECK.
//
// Gathered operands. Eight producer warps copy B with cp.async (16 bytes per thread and
// instruction, into the 128-byte-swizzled layout TMA would write) and hand their completion to the
// stage's mbarrier (cp.async.mbarrier.arrive), so every free stage's copies are in flight at once;
// the MMA thread fences the stage for the async proxy before its MMAs read it. The tile of x or H
// comes by TMA. One thread issues the MMAs into a double-buffered TMEM accumulator; four warps run
// the epilogue. Measured on the 1.5B-like layer (ncu, cold L2): up 103 us, down 106 us; without
// the B copies the same kernels take 64 / 58 us: the generic-proxy shared-memory writes of the
// gather, not the global reads, set the rate (a variant that read nothing took as long).
//
// Every mbarrier wait is bounded (TWELL_ERR_TIMEOUT); on a timeout every role leaves its loop,
// the TMA copies and MMAs in flight are waited for (bounded) and TMEM is freed.
#include <cuda_fp16.h>

#include "twell_common.cuh"

namespace twell {
namespace tu {

constexpr int kTok = 128;          // tokens per tile (MMA M)
constexpr int kBN = 256;           // MMA N
constexpr int kBK = 64;            // k-block: 128 bytes of 16-bit elements
constexpr int kStages = 4;
constexpr int kGatherWarps = 8;
constexpr int kGather = 32 * kGatherWarps;
constexpr int kThreads = 32 * 6 + kGather;  // TMA, MMA, 4 epilogue, 8 gather warps
constexpr uint32_t kABytes = kTok * kBK * 2;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;   // 32 KB
constexpr size_t kSmem = 1024 + kStages * (kABytes + kBBytes) + 256;  // tiles, then the barriers
constexpr uint32_t kTmemCols = 2 * kBN;

struct Args {
    int N, d, f, fpad, n_mt, fw;
    const int32_t* ucnt;   // [n_mt] |U_m|
    const int32_t* ulist;  // [n_mt, f] U_m ascending (first |U_m| entries)
    int32_t* status;
    uint64_t wait_ns;
    // up
    const __nv_bfloat16* Wu;  // [f, d]
    const int2* work;         // up work units (m, N-block)
    const int32_t* n_work;
    const uint32_t* kmask;  // [N, kw] per row: its kept union positions
    int kw;
    __half* H;              // [N, fpad]: a at kept positions, then h
    // down
    const __half* Wd16;  // [f, d]
    __nv_bfloat16* y;    // [N, d]
};

// ------------------------------------------------------------------------------------------
// 1. Union of the kept units of each 128-token tile, in two kernels.
// (a) One warp per token row sets the bits of the row's kept units in its tile's bitmap over d_ff
//     (global, zeroed before the launch): lanes take column tiles, read the tile's count and its
//     in-tile indices 16 at a time.
__global__ void __launch_bounds__(256) union_bits_kernel(const uint16_t* __restrict__ cnt,
                                                         const uint8_t* __restrict__ idx, int N, int f, int T, int nt,
                                                         int fw, uint32_t* __restrict__ bits, int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= N) return;
    uint32_t* bm = bits + static_cast<size_t>(r / kTok) * fw;
    for (int t = lane; t < nt; t += 32) {
        const size_t rt = static_cast<size_t>(r) * nt + t;
        int c = cnt[rt];
        if (c > T) {
            report(status, TWELL_ERR_DEVICE_CHECK);
            c = 0;
        }
        const uint8_t* ir = idx + rt * T;  // the slot holds T >= 64 bytes, 64-byte aligned
        for (int k0 = 0; k0 < c; k0 += 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(ir + k0);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                if (k0 + e < c) {
                    const int i = (wv[e >> 2] >> (8 * (e & 3))) & 0xff;
                    const int j = t * T + i;
                    if (i >= T || j >= f) report(status, TWELL_ERR_DEVICE_CHECK);
                    else atomicOr(&bm[j >> 5], 1u << (j & 31));
                }
            }
        }
    }
}

// (b) One CTA per tile: a block scan of the bitmap words' popcounts gives each word's rank offset;
//     every set bit writes its unit into the ascending list U_m at its rank; |U_m| is the total.
constexpr int kPrefixThreads = 256;
__global__ void __launch_bounds__(kPrefixThreads) union_prefix_kernel(const uint32_t* __restrict__ bits, int f, int fw,
                                                                      int32_t* __restrict__ wpre,
                                                                      int32_t* __restrict__ ulist,
                                                                      int32_t* __restrict__ ucnt)
{
    __shared__ int32_t s_warp[kPrefixThreads / 32];
    const int m = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t* bm = bits + static_cast<size_t>(m) * fw;
    const int per = (fw + kPrefixThreads - 1) / kPrefixThreads;
    const int w0 = threadIdx.x * per, w1 = min(fw, w0 + per);
    int run = 0;
    for (int w = w0; w < w1; ++w) run += __popc(bm[w]);
    int inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    int base = 0, tot = 0;
    for (int w = 0; w < kPrefixThreads / 32; ++w) {
        if (w < warp) base += s_warp[w];
        tot += s_warp[w];
    }
    int pre = base + inc - run;
    int32_t* ul = ulist + static_cast<size_t>(m) * f;
    for (int w = w0; w < w1; ++w) {
        const uint32_t b = bm[w];
        wpre[static_cast<size_t>(m) * fw + w] = pre;
        for (uint32_t v = b; v != 0u; v &= v - 1u) ul[pre++] = 32 * w + __ffs(v) - 1;
    }
    if (threadIdx.x == 0) ucnt[m] = tot;
}

// The up GEMM's work units, (tile, N-block) for every 256 units of every tile's union, tile by tile.
__global__ void __launch_bounds__(1024) union_work_kernel(const int32_t* __restrict__ ucnt, int n_mt,
                                                          int2* __restrict__ work, int32_t* __restrict__ n_work)
{
    __shared__ int32_t s_tot[32];
    __shared__ int32_t s_carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (int m0 = 0; m0 < n_mt; m0 += 1024) {
        const int m = m0 + threadIdx.x;
        const int nb = m < n_mt ? (ucnt[m] + kBN - 1) / kBN : 0;
        int inc = nb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        if (lane == 31) s_tot[warp] = inc;
        __syncthreads();
        int base = s_carry;
        for (int w = 0; w < warp; ++w) base += s_tot[w];
        const int first = base + inc - nb;
        for (int b = 0; b < nb; ++b) work[first + b] = make_int2(m, b);
        __syncthreads();
        if (threadIdx.x == 1023) s_carry = base + inc;
        __syncthreads();
    }
    if (threadIdx.x == 0) *n_work = s_carry;
}

// The gate activations over each tile's union: for every kept entry of row r (unit j at union
// position p = rank of j in the tile's bitmap) H[r, p] = a (fp16) and bit p of the row's keep mask
// kmask[r] (words over the union positions, zeroed here over [0, |U_m| rounded up to 256)) is set.
// H is not cleared: positions the row does not keep hold stale values that the up GEMM's epilogue
// never reads (it selects on the keep mask). One warp per token row; lanes take column tiles.
__global__ void __launch_bounds__(256) tile_expand_kernel(const void* __restrict__ vals, int vals_bf16,
                                                          const uint8_t* __restrict__ idx,
                                                          const uint16_t* __restrict__ cnt, int N, int f, int T,
                                                          int nt, int fpad, int fw, const int32_t* __restrict__ ucnt,
                                                          const uint32_t* __restrict__ bits,
                                                          const int32_t* __restrict__ wpre, __half* __restrict__ H,
                                                          uint32_t* __restrict__ kmask, int kw, int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= N) return;
    const int m = r / kTok;
    const int upad = (ucnt[m] + kBN - 1) / kBN * kBN;
    uint32_t* km = kmask + static_cast<size_t>(r) * kw;
    for (int w = lane; w < upad / 32; w += 32) km[w] = 0u;
    __syncwarp();  // the cleared words are in place before any lane sets a bit in them
    __half* hr = H + static_cast<size_t>(r) * fpad;
    const uint32_t* bm = bits + static_cast<size_t>(m) * fw;
    const int32_t* wp = wpre + static_cast<size_t>(m) * fw;
    bool over = false;
    for (int t = lane; t < nt; t += 32) {
        int c = cnt[static_cast<size_t>(r) * nt + t];
        if (c > T) c = 0;  // recorded by union_bits_kernel
        const size_t e0 = (static_cast<size_t>(r) * nt + t) * T;
        for (int k = 0; k < c; ++k) {
            const int i = idx[e0 + k];
            const int j = t * T + i;
            if (i >= T || j >= f) continue;
            const float av = vals_bf16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(vals)[e0 + k]) << 16)
                                       : static_cast<const float*>(vals)[e0 + k];
            const int w = j >> 5;
            const int p = wp[w] + __popc(bm[w] & ((1u << (j & 31)) - 1u));
            over |= !(fabsf(av) < 65520.0f);
            hr[p] = __float2half_rn(av);
            atomicOr(&km[p >> 5], 1u << (p & 31));
        }
    }
    if (over) report(status, TWELL_ERR_DEVICE_CHECK);
}

// ------------------------------------------------------------------------------------------
// 2./3. Gathered-B tcgen05 GEMM. UP: A = x tile (K-major), B = 256 union rows of Wu_s (K-major);
// DOWN: A = H tile (K-major), B = 64 union rows of Wd16_s per k-block, 256 columns (MN-major).

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Two fp32 values to an fp16 pair (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 16 bytes global -> shared (L2 only, with an L2 eviction policy); src_bytes = 0 writes zeros and
// reads nothing.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
                 "r"(src_bytes), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// The mbarrier receives one arrival (counted against its expected count) once every cp.async this
// thread issued so far has completed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}


// The up GEMM (UP: work units (tile, 256 union positions), K = d_model) and the down GEMM (work
// units (tile, 256 columns of y), K = |U_m|): one persistent launch each, one CTA per SM.
template <bool UP>
__global__ void __launch_bounds__(kThreads, 1) tile_union_gemm_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                      const __grid_constant__ CUtensorMap tmH,
                                                                      const Args g)
{
    constexpr uint32_t IDESC_UP = idesc_bf16_f32(kTok, kBN, false, false);
    constexpr uint32_t IDESC_DN = idesc_f16_f32(kTok, kBN, false, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kABytes;
    uint64_t* fullA = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);  // the A copy of a stage landed
    uint64_t* fullB = fullA + kStages;                                        // every gather thread's copies landed
    uint64_t* empty = fullB + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nbd = (g.d + kBN - 1) / kBN;  // N-blocks of the down GEMM per tile
    constexpr bool phase_up = UP;
    const int units = phase_up ? *g.n_work : g.n_mt * nbd;
    // unit u: up block (m, nb) or down block (m, nb)
    auto unit = [&](int u, int& m, int& nb) -> bool {
        if (phase_up) {
            const int2 w = g.work[u];
            m = w.x;
            nb = w.y;
            return true;
        }
        m = u / nbd;
        nb = u % nbd;
        return false;
    };
    auto kblocks = [&](bool up, int m) { return up ? g.d / kBK : (g.ucnt[m] + kBK - 1) / kBK; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&fullA[s], 1);
            mbar_init(&fullB[s], kGather);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmH);
    }
    if (warp == 1) {
        tmem_alloc<1>(tmem_slot, kTmemCols);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------------ A by TMA
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
                int m, nb;
                const bool up = unit(u, m, nb);
                const int kbs = kblocks(up, m);
                const CUtensorMap* tm = up ? &tmX : &tmH;
                for (int kb = 0; kb < kbs; ++kb) {
                    if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, g.status, g.wait_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&fullA[stage], kABytes);
                    tma_load_2d(sA + stage * kABytes, tm, kb * kBK, m * kTok, &fullA[stage]);
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Wait (bounded, even after an abort) for every copy this thread issued to land, so no
            // TMA write into shared memory is in flight when the CTA exits.
            for (int s = 0; s < kStages; ++s)
                if (issued_mask & (1u << s))
                    wait_bounded(&fullA[s], (issued_phase >> s) & 1u, nullptr, g.status, g.wait_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
                int m, nb;
                const bool up = unit(u, m, nb);
                const int kbs = kblocks(up, m);
                const uint32_t idesc = up ? IDESC_UP : IDESC_DN;
                if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, g.status, g.wait_ns)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                for (int kb = 0; kb < kbs; ++kb) {
                    if (!wait_bounded(&fullA[stage], phase, abort_flag, g.status, g.wait_ns) ||
                        !wait_bounded(&fullB[stage], phase, abort_flag, g.status, g.wait_ns)) {
                        ok = false;
                        break;
                    }
                    // the B stage was written by cp.async (generic proxy): make it visible to the
                    // tensor core's (async proxy) reads
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + stage * kABytes);
                    const uint32_t b_addr = smem_u32(sB + stage * kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t da = desc_sw128(a_addr + k * 32, 16);
                        const uint64_t db = up ? desc_sw128(b_addr + k * 32, 16) : desc_sw128(b_addr + k * 2048, 8192);
                        tc_mma_f16<1>(d_tmem, da, db, idesc, (kb != 0 || k != 0) ? 1u : 0u);
                    }
                    tc_commit<1>(&empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit<1>(&tfull[acc]);  // with kbs == 0 the epilogue stores zeros
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            tc_commit<1>(drain);
            wait_bounded(drain, 0, nullptr, g.status, g.wait_ns);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter
        uint32_t acc = 0, acc_phase = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            int m, nb;
            const bool up = unit(u, m, nb);
            int ok = 1;
            if (lane == 0) ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, g.status, g.wait_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int row = m * kTok + 32 * q + lane;
            const bool row_ok = row < g.N;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * kBN;
            const int n0 = nb * kBN;
            if (up) {
                // H holds a at the row's kept union positions (bits of the keep mask) and stale values
                // elsewhere: h = a * acc where the bit is set, 0 elsewhere, in place; the next chunk's
                // a and mask word are loaded while the current chunk is formed
                const uint4* hp = reinterpret_cast<const uint4*>(g.H + static_cast<size_t>(row) * g.fpad + n0);
                uint4* hw = reinterpret_cast<uint4*>(g.H + static_cast<size_t>(row) * g.fpad + n0);
                const uint32_t* kp = g.kmask + static_cast<size_t>(row) * g.kw + n0 / 32;
                uint4 an[4];
                uint32_t kn = 0u;
                if (row_ok) {
                    kn = kp[0];
#pragma unroll
                    for (int i = 0; i < 4; ++i) an[i] = hp[i];
                }
                bool over = false;
#pragma unroll 1
                for (int ch = 0; ch < kBN / 32; ++ch) {
                    uint4 ac[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) ac[i] = an[i];
                    const uint32_t kc = kn;
                    if (row_ok && ch + 1 < kBN / 32) {
                        kn = kp[ch + 1];
#pragma unroll
                        for (int i = 0; i < 4; ++i) an[i] = hp[4 * (ch + 1) + i];
                    }
                    float v[32];
                    tmem_ld_32x32b_x32(taddr + ch * 32, v);
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t aw[4] = {ac[i].x, ac[i].y, ac[i].z, ac[i].w};
                            uint32_t ow[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c0 = 8 * i + 2 * e;
                                const float2 af = __half22float2(*reinterpret_cast<const __half2*>(&aw[e]));
                                const float h0 = ((kc >> c0) & 1u) ? af.x * v[c0] : 0.0f;
                                const float h1 = ((kc >> (c0 + 1)) & 1u) ? af.y * v[c0 + 1] : 0.0f;
                                over |= !(fabsf(h0) < 65520.0f) || !(fabsf(h1) < 65520.0f);
                                ow[e] = f16x2_bits(h0, h1);
                            }
                            hw[4 * ch + i] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                        }
                    }
                }
                if (over) report(g.status, TWELL_ERR_DEVICE_CHECK);
            } else {
                const bool any = kblocks(false, m) > 0;
                for (int ch = 0; ch < kBN / 32; ++ch) {
                    float v[32];
                    tmem_ld_32x32b_x32(taddr + ch * 32, v);
                    const int col0 = n0 + ch * 32;
                    if (!row_ok || col0 >= g.d) continue;
                    uint4* dst = reinterpret_cast<uint4*>(g.y + static_cast<size_t>(row) * g.d + col0);
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        float f8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) f8[e] = any ? v[i + e] : 0.0f;
                        dst[i / 8] = pack16(f8, static_cast<__nv_bfloat16*>(nullptr));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    } else {
        // ------------------------------------------------------------------ B gather
        // Each thread copies eight 16-byte chunks per stage with cp.async (L2 -> shared, no
        // registers) and hands their completion to the stage's mbarrier (cp.async.mbarrier.arrive:
        // the arrival happens when the thread's copies have landed), so the copies of every free
        // stage are in flight at once. The MMA thread fences them for the async proxy after its wait.
        // Up block: chunk gt % 8 of rows gt / 8 + 32 i (i < 8) of the 256-row tile (a warp instruction
        // covers 4 rows x 128 bytes). Down block: chunk gt % 32 of the 512-byte k-row gt / 32 + 8 i
        // (i < 8) of the 64-row block (a warp instruction covers one k-row's 256 columns); the chunk's
        // 64-column block is (gt % 32) / 8.
        const int gt = threadIdx.x - 32 * 6;  // 0 .. kGather - 1
        const uint64_t pol = policy_evict_last();
        const uint32_t sB0 = smem_u32(sB);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        const int c8 = gt & 7;
        const int r_up = gt >> 3, r_dn = gt >> 5, blk_dn = (gt & 31) >> 3;
        uint32_t off_up[8], off_dn[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int ru = r_up + 32 * i, rd = r_dn + 8 * i;
            off_up[i] = static_cast<uint32_t>(ru) * 128u + ((static_cast<uint32_t>(c8) ^ (ru & 7)) << 4);
            off_dn[i] = static_cast<uint32_t>(blk_dn) * 8192u + static_cast<uint32_t>(rd) * 128u +
                        ((static_cast<uint32_t>(c8) ^ (rd & 7)) << 4);
        }
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            int m, nb;
            const bool up = unit(u, m, nb);
            const int kbs = kblocks(up, m);
            const int U = g.ucnt[m];
            const int32_t* ul = g.ulist + static_cast<size_t>(m) * g.f;
            const int n0 = nb * kBN;
            // up block: the thread's eight weight rows are fixed for the whole unit;
            // down block: the units of its eight k-rows, loaded one k-block ahead of their copies
            const __nv_bfloat16* urow[8];
            int unit_next[8];
            const bool col_ok = up || (n0 + 64 * blk_dn + 8 * c8 < g.d);
            auto units_of = [&](int kb, int (&dst)[8]) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int pp = kb * kBK + r_dn + 8 * i;
                    dst[i] = (col_ok && pp < U) ? ul[pp] : -1;
                }
            };
            if (up) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int pp = n0 + r_up + 32 * i;
                    urow[i] = pp < U ? g.Wu + static_cast<size_t>(ul[pp]) * g.d + 8 * c8 : nullptr;
                }
            } else {
                units_of(0, unit_next);
            }
            for (int kb = 0; kb < kbs; ++kb) {
                int unit_cur[8];
                if (!up) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) unit_cur[i] = unit_next[i];
                    if (kb + 1 < kbs) units_of(kb + 1, unit_next);
                }
                int w = 1;
                if (lane == 0) w = wait_bounded(&empty[stage], phase ^ 1u, abort_flag, g.status, g.wait_ns) ? 1 : 0;
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) {
                    ok = false;
                    break;
                }
                const uint32_t b = sB0 + stage * kBBytes;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (up) {
                        const bool valid = urow[i] != nullptr;
                        cp_async16_zfill(b + off_up[i],
                                         valid ? static_cast<const void*>(urow[i] + kb * kBK) : static_cast<const void*>(g.Wu),
                                         valid ? 16u : 0u, pol);
                    } else {
                        const bool valid = unit_cur[i] >= 0;
                        cp_async16_zfill(b + off_dn[i],
                                         valid ? static_cast<const void*>(g.Wd16 + static_cast<size_t>(unit_cur[i]) * g.d +
                                                                          n0 + 64 * blk_dn + 8 * c8)
                                               : static_cast<const void*>(g.Wd16),
                                         valid ? 16u : 0u, pol);
                    }
                }
                cp_async_arrive_noinc(&fullB[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        cp_async_commit_group();
        cp_async_wait_group<0>();  // no copy into shared memory is in flight when the CTA exits
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<1>(tmem_base, kTmemCols);
}

// Workspace of twell_ffn_tile_union_fwd (byte offsets, 256-byte aligned).
struct TileUnionWs {
    int n_mt = 0, fw = 0, fpad = 0, kw = 0, n_work_cap = 0;
    size_t ucnt = 0, ulist = 0, bits = 0, wpre = 0, work = 0, n_work = 0, kmask = 0, H = 0, total = 0;
    static size_t up(size_t v) { return (v + 255) & ~size_t(255); }
    TileUnionWs(int N, int f)
    {
        n_mt = (N + kTok - 1) / kTok;
        fw = (f + 31) / 32;
        fpad = (f + kBN - 1) / kBN * kBN;
        kw = fpad / 32;
        n_work_cap = n_mt * ((f + kBN - 1) / kBN);
        ucnt = 0;
        ulist = up(static_cast<size_t>(n_mt) * 4);
        bits = ulist + up(static_cast<size_t>(n_mt) * f * 4);
        wpre = bits + up(static_cast<size_t>(n_mt) * fw * 4);
        work = wpre + up(static_cast<size_t>(n_mt) * fw * 4);
        n_work = work + up(static_cast<size_t>(n_work_cap) * 8);
        kmask = n_work + 256;
        H = kmask + up(static_cast<size_t>(N) * kw * 4);
        total = H + up(static_cast<size_t>(N) * fpad * 2);
    }
};

}  // namespace tu
}  // namespace twell

size_t twell_host::tile_union_ws_bytes(int N, int f) { return twell::tu::TileUnionWs(N, f).total; }

using namespace twell_host;

namespace {
template <bool UP>
twell_status launch_tile_union_gemm(const CUtensorMap& tx, const CUtensorMap& th, const twell::tu::Args& g, int max_units,
                                    cudaStream_t s)
{
    using namespace twell::tu;
    DevInfo di;
    if (dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    if (di.max_smem_optin < kSmem) return TWELL_ERR_UNSUPPORTED;
    auto kern = twell::tu::tile_union_gemm_kernel<UP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem)) != cudaSuccess)
        return TWELL_ERR_CUDA;
    const int grid = max_units < di.sm_count ? max_units : di.sm_count;
    if (grid <= 0) return TWELL_OK;
    kern<<<grid, kThreads, kSmem, s>>>(tx, th, g);
    return launch_status();
}
}  // namespace

extern "C" twell_status twell_ffn_tile_union_fwd(const void* x, const void* Wu_s, const void* Wd16_s,
                                                 const twell_packed* a, int32_t N, int32_t d, int32_t f, void* y,
                                                 void* ws, size_t ws_bytes, int32_t* dev_status, void* stream)
{
    using namespace twell::tu;
    if (Wu_s == nullptr || Wd16_s == nullptr || a == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if ((x == nullptr || y == nullptr) && N != 0) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || f > 65535) return TWELL_ERR_INVALID;
    if (d % kBK != 0) return TWELL_ERR_UNSUPPORTED;
    if (!dtype_ok(a->dtype)) return TWELL_ERR_UNSUPPORTED;
    twell_status st = check_packed(a, N, f, a->tile, a->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    const TileUnionWs L(N, f);
    if (ws == nullptr || ws_bytes < L.total) return TWELL_ERR_WORKSPACE;
    const uintptr_t a32 = reinterpret_cast<uintptr_t>(Wu_s) | reinterpret_cast<uintptr_t>(Wd16_s) |
                          reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(ws);
    if (a32 % 32 != 0) return TWELL_ERR_INVALID;  // 32-byte weight loads, 16-byte stores, TMA
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    const int nt = (f + a->tile - 1) / a->tile;

    Args g{};
    g.N = N;
    g.d = d;
    g.f = f;
    g.fpad = L.fpad;
    g.n_mt = L.n_mt;
    g.fw = L.fw;
    g.ucnt = reinterpret_cast<const int32_t*>(w + L.ucnt);
    g.ulist = reinterpret_cast<const int32_t*>(w + L.ulist);
    g.status = dev_status;
    g.wait_ns = wait_limit_ns();
    g.Wu = static_cast<const __nv_bfloat16*>(Wu_s);
    g.work = reinterpret_cast<const int2*>(w + L.work);
    g.n_work = reinterpret_cast<const int32_t*>(w + L.n_work);
    g.kmask = reinterpret_cast<const uint32_t*>(w + L.kmask);
    g.kw = L.kw;
    g.H = reinterpret_cast<__half*>(w + L.H);
    g.Wd16 = static_cast<const __half*>(Wd16_s);
    g.y = static_cast<__nv_bfloat16*>(y);

    uint32_t* bits = reinterpret_cast<uint32_t*>(w + L.bits);
    int32_t* wpre = reinterpret_cast<int32_t*>(w + L.wpre);
    if (cudaMemsetAsync(bits, 0, static_cast<size_t>(L.n_mt) * L.fw * 4, s) != cudaSuccess) return TWELL_ERR_CUDA;
    union_bits_kernel<<<(N + 7) / 8, 256, 0, s>>>(a->cnt, a->idx, N, f, a->tile, nt, L.fw, bits, dev_status);
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    union_prefix_kernel<<<L.n_mt, kPrefixThreads, 0, s>>>(bits, f, L.fw, wpre, reinterpret_cast<int32_t*>(w + L.ulist),
                                                          reinterpret_cast<int32_t*>(w + L.ucnt));
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    union_work_kernel<<<1, 1024, 0, s>>>(g.ucnt, L.n_mt, reinterpret_cast<int2*>(w + L.work),
                                         reinterpret_cast<int32_t*>(w + L.n_work));
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    tile_expand_kernel<<<(N + 7) / 8, 256, 0, s>>>(a->vals, a->dtype == TWELL_BF16 ? 1 : 0, a->idx, a->cnt, N, f,
                                                   a->tile, nt, L.fpad, L.fw, g.ucnt, bits, wpre, g.H,
                                                   reinterpret_cast<uint32_t*>(w + L.kmask), L.kw, dev_status);
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;

    CUtensorMap tx, th;
    st = make_tmap_bf16(&tx, x, d, N, d, kBK, kTok);
    if (st != TWELL_OK) return st;
    st = make_tmap_bf16(&th, w + L.H, L.fpad, N, L.fpad, kBK, kTok);
    if (st != TWELL_OK) return st;
    st = launch_tile_union_gemm<true>(tx, th, g, L.n_work_cap, s);
    if (st != TWELL_OK) return st;
    return launch_tile_union_gemm<false>(tx, th, g, L.n_mt * ((d + kBN - 1) / kBN), s);
}
