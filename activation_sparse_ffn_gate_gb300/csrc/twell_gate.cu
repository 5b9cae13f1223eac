// twell_gate.cu -- gate projection with the TwELL pack in its epilogue.
//
// bf16: the persistent tcgen05 GEMM (twell_gemm.cuh) with the PackTwell epilogue: each epilogue
// thread owns one token row of the 128 x 256 accumulator tile in TMEM, applies ReLU and writes
// the kept entries of every T-wide column tile (values, in-tile indices, count) straight from
// registers -- no dense G, no second pass, no synchronisation between CTAs ([AIM] ¶3;
// [TG] "Вот тут и решает TwELL"; [PUL] ¶3; [TC] §2).
// fp32: a CUDA-core kernel (one warp per row and tile, ballot compaction) for small fp32 layers.
// bf16 batches of at most 16 tokens (decoding): gate_small_kernel (twell_small.cuh).
#include "twell_gemm.cuh"
#include "twell_small.cuh"

namespace twell {

// Gate + pack of at most 16 tokens: the phases of twell_small.cuh on a cluster of two CTAs per
// column tile.
template <int NB, int T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32 * kSmallWarps, 1)
    gate_small_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ Wg, int N, int d, int f,
                      int nt, int vals_f32, void* __restrict__ vals, uint8_t* __restrict__ idx,
                      uint16_t* __restrict__ cnt)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const SmallGateLayout L(NB, T, d);
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int tile = blockIdx.x >> 1;
    small_gate_phase<NB, T>(x, Wg, N, d, f, tile, rank, L, smem, cluster);
    small_pack_phase<NB, T>(N, f, nt, tile, rank, L, smem, cluster, vals_f32, vals, idx, cnt);
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
    // Up to 128 tokens: the transposed kernel (64 units' Wg_s rows per CTA on the MMA's M side, the
    // tokens as its N columns, two CTAs per 128-unit tile): 88 CTAs stream Wg_s at d_ff 5632.
    if (N <= kTransposedMaxN && (T == 64 || T == 128))
        return gate_up_small(x, Wg_s, nullptr, N, d, f, T, out, nullptr, 0, dev_status, s);
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
