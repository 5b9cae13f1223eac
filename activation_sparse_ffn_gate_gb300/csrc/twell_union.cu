// twell_union.cu -- the up and down projections of a dense-enough TwELL layer as two tensor-core
// GEMMs over all of d_ff.
//
// The fused walk (twell_ffn.cu) gathers 2 * d_model weights per kept entry and token; it beats the
// dense layer while tokens keep well under 1% of d_ff. Above that, the union of the units a tile of
// 128 tokens keeps covers most of d_ff (1 - (1 - p)^128 of it: 72% at p = 1%, 99.9% at 5%), so the
// product over all of d_ff is a dense contraction and belongs on the tensor cores ([TC] §3: tensor
// cores take the heavy work, custom sparse kernels the light). Here:
//   1. a is written into H [N, f_pad] (fp16) at each row's kept columns, with a keep mask per row
//      (one bit per column, f_pad = d_ff rounded up to 64); H is not cleared;
//   2. H = (x Wu_s^T) * a: tcgen05 GEMM on SM pairs whose epilogue forms h = a * acc where the mask
//      bit is set (0 elsewhere) and stores it in place as fp16;
//   3. y = H Wd16_s: tcgen05 GEMM on SM pairs over K = f_pad with fp16 operands, B read K-major from
//      Wd16t_s = Wd_s^T converted once to fp16 ([d_model, d_ff], the same values), bf16 y.
// h and a carry 11 significant bits (fp16); an a or h beyond the fp16 range is recorded as
// TWELL_ERR_DEVICE_CHECK. (The earlier form of this path carried h as a bf16 hi + lo pair, which
// doubled K of the down GEMM.)
//
// twell_ffn_gate_union_fwd starts from x instead of a TwELL: one tcgen05 GEMM on SM pairs computes
// the gate and the up projection of the same 128 units in one tile (the even CTA of the pair loads
// Wg_s rows, the odd CTA Wu_s rows; A = x is shared), and its epilogue packs ReLU(g) into the
// TwELL exactly as twell_gate_pack does and stores h = a * u (fp16, 0 where g <= 0) -- no expansion
// pass, no second read of x, no mask. Step 3 follows as above.
//
// Small batches: with at most 1024 tokens the down GEMM has too few 256 x 256 tiles to occupy the SM
// pairs (8 at 64 tokens and d_model 2048), and each pair would stream a whole 256-row block of
// Wd16t_s. There K = f_pad is split into ks ranges (ks * ceil(N / 256) <= 8), each range a work
// unit that stores an fp32 partial product, and a second kernel adds the partials in range order
// (a fixed order: y does not depend on scheduling) and rounds to bf16.
#include <algorithm>

#include "twell_gemm.cuh"

namespace twell {
namespace {

// One warp per token row: the row's keep-mask words are cleared, then each lane takes column tiles
// and writes a (fp16) at H[r, j] and sets bit j of the mask for every kept entry. A count above the
// tile width, an in-tile index at or beyond T or a column at or beyond f is recorded as
// TWELL_ERR_DEVICE_CHECK and skipped; an a beyond the fp16 range is recorded the same way.
template <typename Ein>
__global__ void __launch_bounds__(256) expand_f16_mask_kernel(const Ein* __restrict__ vals,
                                                              const uint8_t* __restrict__ idx,
                                                              const uint16_t* __restrict__ cnt, int N, int f,
                                                              int f_pad, int T, int nt, __half* __restrict__ H,
                                                              uint32_t* __restrict__ mask, int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= N) return;
    const int mw = f_pad / 32;
    uint32_t* mr = mask + static_cast<size_t>(r) * mw;
    for (int w = lane; w < mw; w += 32) mr[w] = 0u;
    __syncwarp();  // cleared words are in place before any lane sets a bit in them
    __half* hr = H + static_cast<size_t>(r) * f_pad;
    bool bad = false;
    for (int t = lane; t < nt; t += 32) {
        int c = cnt[static_cast<size_t>(r) * nt + t];
        if (c > T) {
            bad = true;
            c = 0;
        }
        const size_t e0 = (static_cast<size_t>(r) * nt + t) * T;
        for (int k = 0; k < c; ++k) {
            const int i = idx[e0 + k];
            const int j = t * T + i;
            if (i >= T || j >= f) {
                bad = true;
                continue;
            }
            const float av = Elem<Ein>::to_f(vals[e0 + k]);
            bad |= !(fabsf(av) < 65520.0f);
            hr[j] = __float2half_rn(av);
            atomicOr(&mr[j >> 5], 1u << (j & 31));
        }
    }
    if (bad) report(status, TWELL_ERR_DEVICE_CHECK);
}

// Most rows whose split partial products the down GEMM stores: ks * ceil(N / 256) <= 8 pairs of
// 128-row tiles, i.e. ks * N <= 2048, and splitting only for N <= 1024.
constexpr int kSplitMaxRows = 2048;
constexpr int kSplitMaxN = 1024;
// Above kSplitMaxN tokens: the down GEMM's last, partial wave of 256 x 256 tiles may be cut into K
// halves (at most this many tiles; two fp32 [256 x 256] partials each)
constexpr int kTailMax = 40;
constexpr size_t kTailTileBytes = 2ull * 256 * 256 * 4;

// y over the tail tiles = bf16(half 0 + half 1), four columns per thread. Launched as a programmatic
// dependent of the down GEMM: it waits for that grid before reading.
__global__ void __launch_bounds__(256) reduce_tail_bf16_kernel(const float* __restrict__ part, int ts, int full,
                                                               int n_tiles, int M, int N,
                                                               __nv_bfloat16* __restrict__ y)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<size_t>(ts) * 256 * 64) return;
    const int tt = static_cast<int>(i / (256 * 64)), lr = static_cast<int>(i / 64 % 256), c4 = static_cast<int>(i % 64);
    const int t = full + tt;
    const int m = 2 * (t / n_tiles) * 128 + lr, n = (t % n_tiles) * 256 + 4 * c4;
    if (m >= M || n >= N) return;
    const float4 a = *reinterpret_cast<const float4*>(part + ((static_cast<size_t>(tt) * 2) * 256 + lr) * 256 + 4 * c4);
    const float4 b = *reinterpret_cast<const float4*>(part + ((static_cast<size_t>(tt) * 2 + 1) * 256 + lr) * 256 + 4 * c4);
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x + b.x, a.y + b.y), hi = __floats2bfloat162_rn(a.z + b.z, a.w + b.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&lo);
    w.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(y + static_cast<size_t>(m) * N + n) = w;
}

// y[i] = bf16(part[0][i] + part[1][i] + ... + part[ks - 1][i]) for four elements per thread.
// Launched as a programmatic dependent of the down GEMM: it waits for that grid before reading.
__global__ void __launch_bounds__(256) reduce_splits_bf16_kernel(const float* __restrict__ part, int ks, size_t n,
                                                                 __nv_bfloat16* __restrict__ y)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t i = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
    if (i >= n) return;
    float4 a = *reinterpret_cast<const float4*>(part + i);
    for (int sp = 1; sp < ks; ++sp) {
        const float4 b = *reinterpret_cast<const float4*>(part + static_cast<size_t>(sp) * n + i);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&lo);
    w.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(y + i) = w;
}

inline size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

// bytes of the split partials a call may need: none up to kDownSmallMaxN tokens (the down product
// adds its partials on chip), K ranges up to kSplitMaxN tokens, the tail tiles' K halves above
inline size_t split_bytes(int N, int d)
{
    if (N <= twell_host::kDownSmallMaxN) return 0;
    return N <= kSplitMaxN ? up256(static_cast<size_t>(kSplitMaxRows) * d * 4) : up256(kTailMax * kTailTileBytes);
}

struct UnionWs {
    int f_pad = 0;
    size_t mask = 0, h = 0, part = 0, total = 0;
    UnionWs(int N, int d, int f)
    {
        f_pad = (f + 63) / 64 * 64;
        mask = 0;
        h = up256(static_cast<size_t>(N) * (f_pad / 32) * 4);
        part = h + up256(static_cast<size_t>(N) * f_pad * 2);
        total = part + split_bytes(N, d);
    }
};

}  // namespace
}  // namespace twell

size_t twell_host::union_ws_bytes(int N, int d, int f) { return twell::UnionWs(N, d, f).total; }

size_t twell_host::gate_union_ws_bytes(int N, int d, int f)
{
    return twell::up256(static_cast<size_t>(N) * ((f + 63) / 64 * 64) * 2) + twell::split_bytes(N, d);
}

using namespace twell_host;

namespace {

// Ranges K is split into for the down GEMM: enough work units for half the SM pairs or more, at
// least four k-blocks per range, ks * ceil(N / 256) <= 8; 1 above kSplitMaxN tokens.
int union_down_splits(int N, int d, int fp)
{
    if (N > twell::kSplitMaxN) return 1;
    DevInfo di;
    if (dev_info(&di) != TWELL_OK) return 1;
    const int pairs = di.sm_count / 2;
    const int m_pairs = (N + 255) / 256, n_tiles = (d + 255) / 256;
    const int units = m_pairs * n_tiles;
    if (2 * units >= pairs) return 1;
    int ks = (pairs + units - 1) / units;
    ks = std::min(ks, twell::kSplitMaxRows / 256 / m_pairs);
    ks = std::min(ks, fp / twell::kBK / 4);
    return std::max(ks, 1);
}

// y = H Wd16t_s^T over K = f_pad: A = H [N, f_pad] fp16, B = Wd16t_s [d, f] fp16 K-major (columns
// f .. f_pad read as zeros by TMA), bf16 y, on SM pairs; for small batches split along K into fp32
// partials at `part` (split_bytes(N, d) bytes), added in order by reduce_splits_bf16_kernel.
twell_status union_down(const __half* H, const void* Wd16t_s, int N, int d, int f, int fp, void* y, float* part,
                        int32_t* dev_status, cudaStream_t s)
{
    if (N <= kDownSmallMaxN) return down_small(H, Wd16t_s, N, d, f, fp, y, dev_status, s);
    const int ks = union_down_splits(N, d, fp);
    twell::GemmArgs g2{};
    g2.M = N;
    g2.N = d;
    g2.K = fp;
    g2.ldo = d;
    g2.status = dev_status;
    g2.pdl = 1;  // its prologue overlaps the producing GEMM's last wave
    const GemmOperand A{H, N, fp, fp}, B{Wd16t_s, d, f, f};
    if (ks <= 1) {
        g2.out = y;
        if (N > twell::kSplitMaxN) {  // the partial last wave in K halves, added by reduce_tail_bf16_kernel
            g2.tail_split = -twell::kTailMax;
            g2.tail_part = part;
        }
        int ts = 0;
        twell_status st = launch_gemm<256, false, false, twell::Epi::StoreBF16, true, true>(A, B, nullptr, g2, s, &ts);
        if (st != TWELL_OK || ts == 0) return st;
        const int n_tiles = (d + 255) / 256, tiles = ((N + 255) / 256) * n_tiles;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(static_cast<unsigned>((static_cast<size_t>(ts) * 256 * 64 + 255) / 256));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, twell::reduce_tail_bf16_kernel, static_cast<const float*>(part), ts, tiles - ts,
                               n_tiles, N, d, static_cast<__nv_bfloat16*>(y)) != cudaSuccess)
            return TWELL_ERR_CUDA;
        return launch_status();
    }
    g2.out = part;
    g2.k_splits = ks;
    g2.split_stride = static_cast<int64_t>(N) * d;
    twell_status st = launch_gemm<256, false, false, twell::Epi::StoreF32, true, true>(A, B, nullptr, g2, s);
    if (st != TWELL_OK) return st;
    const size_t n = static_cast<size_t>(N) * d;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>((n / 4 + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, twell::reduce_splits_bf16_kernel, static_cast<const float*>(part), ks, n,
                           static_cast<__nv_bfloat16*>(y)) != cudaSuccess)
        return TWELL_ERR_CUDA;
    return launch_status();
}

}  // namespace

extern "C" twell_status twell_ffn_union_fwd(const void* x, const void* Wu_s, const void* Wd16t_s, const twell_packed* a,
                                            int32_t N, int32_t d, int32_t f, twell_dtype dtype, void* y, void* ws,
                                            size_t ws_bytes, int32_t* dev_status, void* stream)
{
    if (Wu_s == nullptr || Wd16t_s == nullptr || a == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if ((x == nullptr || y == nullptr) && N != 0) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0 || f % 8 != 0) return TWELL_ERR_INVALID;
    if (dtype != TWELL_BF16 || !dtype_ok(a->dtype)) return TWELL_ERR_UNSUPPORTED;
    twell_status st = check_packed(a, N, f, a->tile, a->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    const twell::UnionWs L(N, d, f);
    if (ws == nullptr || ws_bytes < L.total) return TWELL_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(Wu_s) || !aligned16(Wd16t_s) || !aligned16(y) || !aligned16(ws))
        return TWELL_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* M = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + L.mask);
    __half* H = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) + L.h);
    const int T = a->tile, nt = (f + T - 1) / T;
    const int fp = L.f_pad;
    // 1. a at the kept columns of H, keep masks
    const unsigned blocks = static_cast<unsigned>((N + 7) / 8);
    if (a->dtype == TWELL_BF16)
        twell::expand_f16_mask_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(a->vals), a->idx, a->cnt, N, f, fp, T, nt, H, M, dev_status);
    else
        twell::expand_f16_mask_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float*>(a->vals), a->idx,
                                                                    a->cnt, N, f, fp, T, nt, H, M, dev_status);
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    // 2. h = (x Wu_s^T) * a in place (columns f .. f_pad of Wu_s read as zeros, their mask bits clear)
    twell::GemmArgs g{};
    g.M = N;
    g.N = fp;
    g.K = d;
    g.out = H;
    g.ldo = fp;
    g.aux = H;
    g.ldaux = fp;
    g.mask = M;
    g.ldmask = fp / 32;
    g.status = dev_status;
    st = launch_gemm<256, false, false, twell::Epi::MulMaskF16, true>(GemmOperand{x, N, d, d},
                                                                      GemmOperand{Wu_s, f, d, d}, nullptr, g, s);
    if (st != TWELL_OK) return st;
    // 3. y = H Wd16_s over K = f_pad
    return union_down(H, Wd16t_s, N, d, f, fp, y, reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.part),
                      dev_status, s);
}

extern "C" twell_status twell_ffn_gate_union_fwd(const void* x, const void* Wg_s, const void* Wu_s,
                                                 const void* Wd16t_s, int32_t N, int32_t d, int32_t f, int32_t T,
                                                 twell_dtype dtype, const twell_packed* out, void* y, void* ws,
                                                 size_t ws_bytes, int32_t* dev_status, void* stream)
{
    if (Wg_s == nullptr || Wu_s == nullptr || Wd16t_s == nullptr || out == nullptr || dev_status == nullptr)
        return TWELL_ERR_INVALID;
    if ((x == nullptr || y == nullptr) && N != 0) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0 || f % 8 != 0) return TWELL_ERR_INVALID;
    if (dtype != TWELL_BF16 || !dtype_ok(out->dtype) || (T != 64 && T != 128)) return TWELL_ERR_UNSUPPORTED;
    twell_status st = check_packed(out, N, f, T, out->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    if (ws == nullptr || ws_bytes < gate_union_ws_bytes(N, d, f)) return TWELL_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(Wg_s) || !aligned16(Wu_s) || !aligned16(Wd16t_s) || !aligned16(y) ||
        !aligned16(ws))
        return TWELL_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    __half* H = static_cast<__half*>(ws);
    const int fp = (f + 63) / 64 * 64;
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                           twell::up256(static_cast<size_t>(N) * fp * 2));
    if (N <= kTransposedMaxN) {  // weights on the M side of both products
        st = gate_up_small(x, Wg_s, Wu_s, N, d, f, T, out, H, fp, dev_status, s);
        if (st != TWELL_OK) return st;
        return down_small(H, Wd16t_s, N, d, f, fp, y, dev_status, s);
    }
    // 1 + 2. g and u of each 128-unit block in one tile: TwELL of ReLU(g), h = a * u into H
    twell::GemmArgs g{};
    g.M = N;
    g.N = f;
    g.K = d;
    g.out = H;
    g.ldo = fp;
    g.vals_f32 = out->dtype == TWELL_F32 ? 1 : 0;
    g.vals = out->vals;
    g.idx = out->idx;
    g.cnt = out->cnt;
    g.T = T;
    g.nt = (f + T - 1) / T;
    g.status = dev_status;
    g.pdl = 1;  // its prologue overlaps the tail of the kernel before it on the stream
    const GemmOperand Bu{Wu_s, f, d, d};
    st = launch_gemm<256, false, false, twell::Epi::GateUpF16, true>(GemmOperand{x, N, d, d},
                                                                     GemmOperand{Wg_s, f, d, d}, &Bu, g, s);
    if (st != TWELL_OK) return st;
    // 3. y = H Wd16_s over K = f_pad
    return union_down(H, Wd16t_s, N, d, f, fp, y, part, dev_status, s);
}
