// twell_gate.cu -- gate projection with the TwELL pack in its epilogue.
//
// bf16: the persistent tcgen05 GEMM (twell_gemm.cuh) with the PackTwell epilogue: each epilogue
// thread owns one token row of the 128 x 256 accumulator tile in TMEM, applies ReLU and writes
// the kept entries of every T-wide column tile (values, in-tile indices, count) straight from
// registers -- no dense G, no second pass, no synchronisation between CTAs ([AIM] ¶3;
// [TG] "Вот тут и решает TwELL"; [PUL] ¶3; [TC] §2).
// fp32: a CUDA-core kernel (one warp per row and tile, ballot compaction) for small fp32 layers.
// bf16 batches of at most 16 tokens (decoding): gate_small_kernel, below.
#include <cooperative_groups.h>

#include "twell_gemm.cuh"
#include "twell_mma.cuh"

namespace twell {

// Gate + pack for a batch of at most 16 tokens (bf16). The GEMM is a skinny one: Wg_s (d_ff x
// d_model, 23 MB on the 1.5B-like layer) is read once, and with 128 x T tiles only d_ff / T SMs
// stream it. Here a cluster of two CTAs owns one T-wide column tile, each CTA T/2 hidden units,
// so twice as many SMs share the read, and every CTA keeps 128 KB of weight loads in flight:
//   * 16 warps; warp w takes the 16-unit block w % (U/16) and every (16/(U/16))-th 64-element
//     span of d_model; per span each lane loads 32 contiguous bytes of its two units' rows
//     (16-byte read-only loads that skip L1) -- the k order inside a span is permuted the same way
//     for both operands, so the fragments come straight from those loads;
//   * x (padded to 8 or 16 token rows, rows >= N zero) is staged in shared memory once;
//   * products on mma.sync m16n8k16 (units as the 16 rows, tokens as the 8 columns), fp32
//     accumulation; the warps' partial sums over d_model are added in a fixed order, so g does not
//     depend on scheduling;
//   * the two CTAs of the cluster exchange nothing but their g values: after a cluster barrier,
//     CTA c packs tokens c, c + 2, ... over the whole tile, reading the other half from the peer's
//     shared memory (distributed shared memory), in ascending column order, as the tile epilogue.
// An entry is kept iff its fp32 g is > 0, and its value stored as g (fp32) or bf16(g).
constexpr int kSmallWarps = 16;
constexpr int kSmallMaxN = 16;

struct SmallGateLayout {
    size_t x_stride, x, part, g, total;
    __host__ __device__ SmallGateLayout(int NB, int T, int d)
    {
        const int U = T / 2, KS = kSmallWarps / (U / 16);
        x_stride = static_cast<size_t>(d) * 2 + 16;  // 16-byte pad: the 8 token rows fall in different banks
        x = 0;
        part = static_cast<size_t>(8 * NB) * x_stride;
        g = part + static_cast<size_t>(KS) * U * 8 * NB * 4;
        total = g + static_cast<size_t>(U) * 8 * NB * 4;
    }
};

template <int NB, int T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32 * kSmallWarps, 1)
    gate_small_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ Wg, int N, int d, int f,
                      int nt, int vals_f32, void* __restrict__ vals, uint8_t* __restrict__ idx,
                      uint16_t* __restrict__ cnt)
{
    constexpr int U = T / 2;             // hidden units per CTA
    constexpr int MB = U / 16;           // 16-unit blocks per CTA
    constexpr int KS = kSmallWarps / MB;  // warps sharing a block (split of d_model)
    constexpr int NTOK = 8 * NB;
    extern __shared__ __align__(16) uint8_t smem[];
    const SmallGateLayout L(NB, T, d);
    uint8_t* xs = smem + L.x;
    float* part = reinterpret_cast<float*>(smem + L.part);  // [KS][U][NTOK]
    float* gs = reinterpret_cast<float*>(smem + L.g);       // [U][NTOK]
    namespace cgx = cooperative_groups;
    cgx::cluster_group cluster = cgx::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int tile = blockIdx.x >> 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;

    // x rows (zeros past N)
    const int chunks = d / 8;
    for (int i = threadIdx.x; i < NTOK * chunks; i += blockDim.x) {
        const int r = i / chunks, c = i - r * chunks;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < N) v = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(r) * d + c * 8);
        *reinterpret_cast<uint4*>(xs + r * L.x_stride + c * 16) = v;
    }
    __syncthreads();

    const int mb = warp % MB, ks = warp / MB;
    const int ua = tile * T + rank * U + mb * 16 + g, ub = ua + 8;  // this lane's two units
    const bool oka = ua < f, okb = ub < f;
    const __nv_bfloat16* wa = Wg + static_cast<size_t>(oka ? ua : 0) * d + 16 * t;
    const __nv_bfloat16* wb = Wg + static_cast<size_t>(okb ? ub : 0) * d + 16 * t;
    const uint8_t* xg = xs + g * L.x_stride + 32 * t;
    float acc[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = acc[b][2] = acc[b][3] = 0.0f;
    const int nspan = d / 64;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int s0 = ks; s0 < nspan; s0 += 4 * KS) {
        uint4 w[4][4];  // per span: unit a elements 0-7, 8-15; unit b elements 0-7, 8-15
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = s0 + i * KS;
            const bool in = s < nspan;
            w[i][0] = (in && oka) ? ldg_stream16(wa + s * 64) : z;
            w[i][1] = (in && oka) ? ldg_stream16(wa + s * 64 + 8) : z;
            w[i][2] = (in && okb) ? ldg_stream16(wb + s * 64) : z;
            w[i][3] = (in && okb) ? ldg_stream16(wb + s * 64 + 8) : z;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = s0 + i * KS;
            if (s >= nspan) break;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const uint8_t* xp = xg + b * 8 * L.x_stride + s * 128;
                const uint4 x0 = *reinterpret_cast<const uint4*>(xp);
                const uint4 x1 = *reinterpret_cast<const uint4*>(xp + 16);
                // k step q of the span uses words 2q, 2q + 1 of each lane's 32 bytes
                mma_bf16(acc[b], w[i][0].x, w[i][2].x, w[i][0].y, w[i][2].y, x0.x, x0.y);
                mma_bf16(acc[b], w[i][0].z, w[i][2].z, w[i][0].w, w[i][2].w, x0.z, x0.w);
                mma_bf16(acc[b], w[i][1].x, w[i][3].x, w[i][1].y, w[i][3].y, x1.x, x1.y);
                mma_bf16(acc[b], w[i][1].z, w[i][3].z, w[i][1].w, w[i][3].w, x1.z, x1.w);
            }
        }
    }
    // fragment: (unit g, tokens 2t, 2t+1), (unit g + 8, tokens 2t, 2t+1) of block b
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float* pa = part + (static_cast<size_t>(ks) * U + mb * 16 + g) * NTOK + b * 8 + 2 * t;
        pa[0] = acc[b][0];
        pa[1] = acc[b][1];
        pa[8 * NTOK] = acc[b][2];
        pa[8 * NTOK + 1] = acc[b][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < U * NTOK; i += blockDim.x) {
        float v = part[i];
        for (int k = 1; k < KS; ++k) v += part[static_cast<size_t>(k) * U * NTOK + i];
        gs[i] = v;
    }
    cluster.sync();  // both halves of the tile's g are in shared memory

    // pack: warp w of CTA c takes token c + 2 w
    const int r = rank + 2 * warp;
    if (warp < NTOK / 2 && r < N) {
        const float* half[2] = {cluster.map_shared_rank(gs, 0), cluster.map_shared_rank(gs, 1)};
        const size_t slot = (static_cast<size_t>(r) * nt + tile) * T;
        int c = 0;
#pragma unroll
        for (int k0 = 0; k0 < T; k0 += 32) {
            const int k = k0 + lane;
            const float v = half[k / U][(k % U) * NTOK + r];
            const bool keep = tile * T + k < f && v > 0.0f;
            const unsigned m = __ballot_sync(0xffffffffu, keep);
            const int pos = c + __popc(m & ((1u << lane) - 1u));
            if (keep) {
                if (vals_f32) static_cast<float*>(vals)[slot + pos] = v;
                else static_cast<__nv_bfloat16*>(vals)[slot + pos] = __float2bfloat16_rn(v);
                idx[slot + pos] = static_cast<uint8_t>(k);
            }
            c += __popc(m);
        }
        if (lane == 0) cnt[static_cast<size_t>(r) * nt + tile] = static_cast<uint16_t>(c);
    }
    cluster.sync();  // the peer's g stays in place until both CTAs have read it
}

template <int NB, int T>
static twell_status launch_gate_small(const __nv_bfloat16* x, const __nv_bfloat16* Wg, int N, int d, int f, int nt,
                                      const twell_packed* out, cudaStream_t s)
{
    const SmallGateLayout L(NB, T, d);
    auto kern = gate_small_kernel<NB, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total)) !=
        cudaSuccess)
        return TWELL_ERR_CUDA;
    kern<<<2 * nt, 32 * kSmallWarps, L.total, s>>>(x, Wg, N, d, f, nt, out->dtype == TWELL_F32 ? 1 : 0, out->vals,
                                                   out->idx, out->cnt);
    return twell_host::launch_status();
}

template <int NB>
static twell_status run_gate_small(const __nv_bfloat16* x, const __nv_bfloat16* Wg, int N, int d, int f, int T,
                                   int nt, const twell_packed* out, cudaStream_t s)
{
    switch (T) {
    case 64: return launch_gate_small<NB, 64>(x, Wg, N, d, f, nt, out, s);
    case 128: return launch_gate_small<NB, 128>(x, Wg, N, d, f, nt, out, s);
    case 256: return launch_gate_small<NB, 256>(x, Wg, N, d, f, nt, out, s);
    default: return TWELL_ERR_UNSUPPORTED;
    }
}

// fp32 gate + pack: warp w handles (row r, tile t); lanes take 32 columns at a time.
__global__ void gate_pack_f32_kernel(const float* __restrict__ x, const float* __restrict__ Wg, int N, int d,
                                     int f, int T, int nt, float* __restrict__ vals, uint8_t* __restrict__ idx,
                                     uint16_t* __restrict__ cnt)
{
    const int lane = threadIdx.x & 31;
    const long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= static_cast<long long>(N) * nt) return;
    const int r = static_cast<int>(w / nt), t = static_cast<int>(w % nt);
    const float* xr = x + static_cast<size_t>(r) * d;
    const size_t slot = (static_cast<size_t>(r) * nt + t) * T;
    int c = 0;
    for (int ch = 0; ch < T; ch += 32) {
        const int k = ch + lane;
        const int j = t * T + k;
        float g = 0.0f;
        if (j < f) {
            const float* wr = Wg + static_cast<size_t>(j) * d;
            for (int i = 0; i < d; ++i) g = fmaf(xr[i], wr[i], g);
        }
        const bool keep = j < f && g > 0.0f;
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        const int pos = c + __popc(m & ((1u << lane) - 1u));
        if (keep) {
            vals[slot + pos] = g;
            idx[slot + pos] = static_cast<uint8_t>(k);
        }
        c += __popc(m);
    }
    if (lane == 0) cnt[static_cast<size_t>(r) * nt + t] = static_cast<uint16_t>(c);
}

}  // namespace twell

using namespace twell_host;

extern "C" twell_status twell_gate_pack(const void* x, const void* Wg_s, int32_t N, int32_t d, int32_t f, int32_t T,
                                        twell_dtype dtype, const twell_packed* out, void* ws, size_t ws_bytes,
                                        int32_t* dev_status, void* stream)
{
    (void)ws;
    (void)ws_bytes;
    if (Wg_s == nullptr || dev_status == nullptr || (x == nullptr && N != 0)) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0) return TWELL_ERR_INVALID;
    if (!dtype_ok(dtype) || out == nullptr || !dtype_ok(out->dtype)) return TWELL_ERR_UNSUPPORTED;
    // fp32 inputs pack fp32 values; bf16 inputs pack either bf16 or fp32 values
    if (dtype == TWELL_F32 && out->dtype != TWELL_F32) return TWELL_ERR_INVALID;
    twell_status st = check_packed(out, N, f, T, out->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    if (!aligned16(x) || !aligned16(Wg_s)) return TWELL_ERR_INVALID;
    const int nt = (f + T - 1) / T;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == TWELL_F32) {
        const long long warps = static_cast<long long>(N) * nt;
        const int per_block = 8;
        const long long blocks = (warps + per_block - 1) / per_block;
        if (blocks > 0x7fffffffLL) return TWELL_ERR_UNSUPPORTED;
        twell::gate_pack_f32_kernel<<<static_cast<unsigned>(blocks), per_block * 32, 0, s>>>(
            static_cast<const float*>(x), static_cast<const float*>(Wg_s), N, d, f, T, nt,
            static_cast<float*>(out->vals), out->idx, out->cnt);
        return launch_status();
    }
    if (N <= twell::kSmallMaxN && d % 64 == 0 && d <= 4096 && (T == 64 || T == 128 || T == 256)) {
        using bf = __nv_bfloat16;
        const bf* xb = static_cast<const bf*>(x);
        const bf* wb = static_cast<const bf*>(Wg_s);
        return N <= 8 ? twell::run_gate_small<1>(xb, wb, N, d, f, T, nt, out, s)
                      : twell::run_gate_small<2>(xb, wb, N, d, f, T, nt, out, s);
    }
    twell::GemmArgs g{};
    g.M = N;
    g.N = f;
    g.K = d;
    g.vals_f32 = out->dtype == TWELL_F32 ? 1 : 0;
    g.vals = out->vals;
    g.idx = out->idx;
    g.cnt = out->cnt;
    g.T = T;
    g.nt = nt;
    g.status = dev_status;
    GemmOperand A{x, N, d, d};
    GemmOperand B{Wg_s, f, d, d};
    // A small batch (decoding a few tokens) fills one or two 128-row tiles: 128 x T tiles on single
    // SMs spread d_ff over more SMs and pad M to 128 rows instead of 256 (the 256 x 256 pair tiles
    // left the decode gate tensor-bound on padding rows, 44 SMs busy at N = 8).
    if (N <= 256) {
        if (T == 64) return launch_gemm<64, false, false, twell::Epi::PackTwell>(A, B, nullptr, g, s);
        if (T == 128) return launch_gemm<128, false, false, twell::Epi::PackTwell>(A, B, nullptr, g, s);
    }
    return launch_gemm<256, false, false, twell::Epi::PackTwell, true>(A, B, nullptr, g, s);
}

extern "C" twell_status twell_gate_gemm(const void* x, const void* Wg_s, int32_t N, int32_t d, int32_t f,
                                        float* G_out, int32_t* dev_status, void* stream)
{
    if (x == nullptr || Wg_s == nullptr || G_out == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0 || f % 4 != 0) return TWELL_ERR_INVALID;
    if (!aligned16(x) || !aligned16(Wg_s) || !aligned16(G_out)) return TWELL_ERR_INVALID;
    if (N == 0) return TWELL_OK;
    twell::GemmArgs g{};
    g.M = N;
    g.N = f;
    g.K = d;
    g.out = G_out;
    g.ldo = f;
    g.status = dev_status;
    GemmOperand A{x, N, d, d};
    GemmOperand B{Wg_s, f, d, d};
    return launch_gemm<256, false, false, twell::Epi::StoreF32, true>(A, B, nullptr, g, static_cast<cudaStream_t>(stream));
}
