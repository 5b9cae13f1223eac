// twell_union.cu -- the up and down projections of a dense-enough TwELL layer as two tensor-core
// GEMMs over all of d_ff.
//
// The fused walk (twell_ffn.cu) gathers 2 * d_model weights per kept entry and token; it beats
// the dense layer while tokens keep well under 1% of d_ff. Above that, the union of the units a
// tile of 128 tokens keeps covers most of d_ff (1 - (1 - p)^128 of it: 72% at p = 1%, 99.9% at 5%),
// so the product over the union is a dense contraction and belongs on the tensor cores ([TC] §3:
// tensor cores take the heavy work, custom sparse kernels the light). Here:
//   1. the TwELL is expanded to a dense bf16 a = ReLU(G) [N, f_pad] (zeros where nothing was kept;
//      f_pad = d_ff rounded up to 64);
//   2. H = (x Wu_s^T) * a: tcgen05 GEMM on SM pairs whose epilogue multiplies the fp32 accumulator
//      by a and stores h as two bf16 terms, [hi | lo] with hi = bf16(h), lo = bf16(h - hi)
//      ([N, 2 f_pad]), so h is carried to ~16 significant bits as in the walk;
//   3. y = [hi | lo] [Wd_s ; Wd_s]: tcgen05 GEMM over K = 2 f_pad (Wd_s read MN-major, twice), bf16 y.
// a is rounded to bf16 (exact for bf16 TwELL values). With h rounded once to bf16 instead, the
// max-abs error reached 2.2e-2 x RMS of the output row on a 5%-dense layer, over the 2e-2 bound.
#include "twell_gemm.cuh"

namespace twell {
namespace {

// One warp per (token row, column tile): the tile's columns of the dense row (pitch f_pad, the
// last tile's up to f_pad) get 0, then the kept entries their value (rounded to bf16). A count
// above the tile width or a column at or beyond f is recorded as TWELL_ERR_DEVICE_CHECK and skipped.
template <typename Ein>
__global__ void expand_bf16_kernel(const Ein* __restrict__ vals, const uint8_t* __restrict__ idx,
                                   const uint16_t* __restrict__ cnt, int N, int f, int f_pad, int T, int nt,
                                   __nv_bfloat16* __restrict__ dense, int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= static_cast<long long>(N) * nt) return;
    const int r = static_cast<int>(w / nt), t = static_cast<int>(w % nt);
    __nv_bfloat16* out = dense + static_cast<size_t>(r) * f_pad;
    for (int k = lane; k < T; k += 32) {
        const int j = t * T + k;
        if (j < f_pad) out[j] = __float2bfloat16_rn(0.0f);
    }
    __syncwarp();
    int c = cnt[static_cast<size_t>(r) * nt + t];
    if (c > T) {
        if (lane == 0) report(status, TWELL_ERR_DEVICE_CHECK);
        c = T;
    }
    const size_t slot = (static_cast<size_t>(r) * nt + t) * T;
    for (int k = lane; k < c; k += 32) {
        const int j = t * T + idx[slot + k];
        if (j < f) out[j] = __float2bfloat16_rn(Elem<Ein>::to_f(vals[slot + k]));
        else report(status, TWELL_ERR_DEVICE_CHECK);
    }
}

struct UnionWs {
    int f_pad = 0;
    size_t a = 0, h = 0, total = 0;
    static size_t up(size_t v) { return (v + 255) & ~size_t(255); }
    UnionWs(int N, int f)
    {
        f_pad = (f + 63) / 64 * 64;
        a = 0;
        h = up(static_cast<size_t>(N) * f_pad * 2);
        total = h + up(static_cast<size_t>(N) * 2 * f_pad * 2);
    }
};

}  // namespace
}  // namespace twell

size_t twell_host::union_ws_bytes(int N, int f) { return twell::UnionWs(N, f).total; }

using namespace twell_host;

extern "C" twell_status twell_ffn_union_fwd(const void* x, const void* Wu_s, const void* Wd_s, const twell_packed* a,
                                            int32_t N, int32_t d, int32_t f, twell_dtype dtype, void* y, void* ws,
                                            size_t ws_bytes, int32_t* dev_status, void* stream)
{
    if (Wu_s == nullptr || Wd_s == nullptr || a == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if ((x == nullptr || y == nullptr) && N != 0) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0 || f % 8 != 0) return TWELL_ERR_INVALID;
    if (dtype != TWELL_BF16 || !dtype_ok(a->dtype)) return TWELL_ERR_UNSUPPORTED;
    twell_status st = check_packed(a, N, f, a->tile, a->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    const twell::UnionWs L(N, f);
    if (ws == nullptr || ws_bytes < L.total) return TWELL_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(Wu_s) || !aligned16(Wd_s) || !aligned16(y) || !aligned16(ws))
        return TWELL_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    using bf = __nv_bfloat16;
    bf* A = reinterpret_cast<bf*>(static_cast<uint8_t*>(ws) + L.a);
    bf* H = reinterpret_cast<bf*>(static_cast<uint8_t*>(ws) + L.h);
    const int T = a->tile, nt = (f + T - 1) / T;
    // 1. dense a
    const long long warps = static_cast<long long>(N) * nt;
    const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
    const int fp = L.f_pad;
    if (a->dtype == TWELL_BF16)
        twell::expand_bf16_kernel<bf><<<blocks, 256, 0, s>>>(static_cast<const bf*>(a->vals), a->idx, a->cnt, N, f, fp,
                                                             T, nt, A, dev_status);
    else
        twell::expand_bf16_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float*>(a->vals), a->idx, a->cnt, N,
                                                                f, fp, T, nt, A, dev_status);
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    // 2. [hi | lo] of H = (x Wu_s^T) * a (columns f .. f_pad of Wu_s read as zeros)
    twell::GemmArgs g{};
    g.M = N;
    g.N = fp;
    g.K = d;
    g.out = H;
    g.ldo = 2 * fp;
    g.lo_offset = fp;
    g.aux = A;
    g.ldaux = fp;
    g.status = dev_status;
    st = launch_gemm<256, false, false, twell::Epi::MulHiLoBF16, true>(GemmOperand{x, N, d, d},
                                                                       GemmOperand{Wu_s, f, d, d}, nullptr, g, s);
    if (st != TWELL_OK) return st;
    // 3. y = [hi | lo] [Wd_s ; Wd_s]
    twell::GemmArgs g2{};
    g2.M = N;
    g2.N = d;
    g2.K = 2 * fp;
    g2.kb_split = fp / 64;
    g2.out = y;
    g2.ldo = d;
    g2.status = dev_status;
    const GemmOperand Bd{Wd_s, f, d, d};
    return launch_gemm<256, false, true, twell::Epi::StoreBF16>(GemmOperand{H, N, 2 * fp, 2 * fp}, Bd, &Bd, g2, s);
}
