// twell_decode.cu -- the whole sparse FFN of a batch of at most 16 tokens (decoding) in two
// launches: y = (ReLU(x Wg_s^T) * (x Wu_s^T)) Wd_s with the gate activations packed as TwELL
// ([AIM] ¶3; [TG] "Инференс"; [PUL] ¶3; [TC] §2).
//
// At a few tokens every step of the two-call path (gate + pack, then the walk) is a chain of
// launches and memory round trips: the walk alone costs ~25 us at one token, for ~30 nonzeros.
// The TwELL makes the walk separable by column tile, y_r = sum over tiles of sum over the tile's
// kept units, so the CTAs that compute a tile's gate values can walk that tile's nonzeros at once:
//   1. decode_small_kernel, a cluster of two CTAs per T-wide column tile, each CTA T/2 units: the
//      gate and the pack of twell_small.cuh (the same TwELL, bit for bit, as twell_gate_pack), then
//      over the CTA's own units: the units some token keeps are listed in ascending order; one warp
//      per listed unit reads its row of Wu_s and forms u = x_r . Wu_s[j] for each token keeping it
//      (fp32, lanes in a fixed order, then a butterfly), h = a * u with a the packed value; then the
//      CTA's threads, four columns each, add h * Wd_s[j] over the listed units in ascending order
//      (fp32) and store one fp32 partial row per token that keeps any of the CTA's units, with a
//      flag per (CTA, token) saying whether it did;
//   2. decode_reduce_kernel adds, per token and column, the flagged partial rows in a fixed order
//      and stores y in bf16. y does not depend on scheduling.
#include "twell_small.cuh"

namespace twell {
namespace {

constexpr int kDecodeChunks = 8;  // 16-byte chunks of a Wu_s row a lane has in flight

// The gate layout, then the kept-unit list [U] (local unit index), the units' token masks [U], the
// number of listed units and the CTA's token mask. h [U][8 NB] reuses the partial-g area, which is
// free once g is summed.
struct DecodeLayout {
    SmallGateLayout G;
    size_t h, list, mask, meta, total;
    __host__ __device__ DecodeLayout(int NB, int T, int d) : G(NB, T, d)
    {
        h = G.part;
        list = (G.total + 15) & ~size_t(15);
        mask = list + static_cast<size_t>(T / 2) * 4;
        meta = mask + static_cast<size_t>(T / 2) * 4;
        total = meta + 16;
    }
};

struct DecodeWs {
    size_t flags = 0, part = 0, total = 0;
    static size_t up(size_t v) { return (v + 255) & ~size_t(255); }
    DecodeWs(int N, int d, int f, int T)
    {
        const size_t ncta = 2 * static_cast<size_t>((f + T - 1) / T);
        flags = 0;
        part = up(ncta * N * 4);
        total = part + up(ncta * N * static_cast<size_t>(d) * 4);
    }
};

__device__ __forceinline__ float dot8(const uint4& w, const uint4& x)
{
    const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&w);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&x);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __bfloat1622float2(a[i]);
        const float2 q = __bfloat1622float2(b[i]);
        s = fmaf(p.x, q.x, s);
        s = fmaf(p.y, q.y, s);
    }
    return s;
}

template <int NB, int T>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32 * kSmallWarps, 1)
    decode_small_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ Wg,
                        const __nv_bfloat16* __restrict__ Wu, const __nv_bfloat16* __restrict__ Wd, int N, int d,
                        int f, int nt, int vals_f32, void* __restrict__ vals, uint8_t* __restrict__ idx,
                        uint16_t* __restrict__ cnt, float* __restrict__ part_y, int* __restrict__ flags)
{
    constexpr int U = T / 2;
    constexpr int NTOK = 8 * NB;
    extern __shared__ __align__(16) uint8_t smem[];
    const DecodeLayout L(NB, T, d);
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int tile = blockIdx.x >> 1;
    const int u_base = tile * T + rank * U;  // first unit of this CTA
    // the reduction kernel may be scheduled now: it waits for this grid at its griddepcontrol.wait
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    small_gate_phase<NB, T>(x, Wg, N, d, f, tile, rank, L.G, smem, cluster);
    small_pack_phase<NB, T>(N, f, nt, tile, rank, L.G, smem, cluster, vals_f32, vals, idx, cnt);

    const float* gs = reinterpret_cast<const float*>(smem + L.G.g);  // [U][NTOK]
    float* hs = reinterpret_cast<float*>(smem + L.h);                // [U][NTOK]
    int* list = reinterpret_cast<int*>(smem + L.list);
    unsigned* umask = reinterpret_cast<unsigned*>(smem + L.mask);
    int* meta = reinterpret_cast<int*>(smem + L.meta);  // [0] listed units, [1] token mask
    const uint8_t* xs = smem + L.G.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // h = 0; the units some token keeps, ascending, with the tokens that keep each
    for (int i = threadIdx.x; i < U * NTOK; i += blockDim.x) hs[i] = 0.0f;
    if (warp == 0) {
        int n = 0;
        unsigned tm = 0u;
        for (int u0 = 0; u0 < U; u0 += 32) {
            const int u = u0 + lane;
            unsigned m = 0u;
            if (u < U && u_base + u < f) {
                for (int r = 0; r < N; ++r)
                    if (gs[u * NTOK + r] > 0.0f) m |= 1u << r;
            }
            const unsigned b = __ballot_sync(0xffffffffu, m != 0u);
            if (m != 0u) {
                const int pos = n + __popc(b & ((1u << lane) - 1u));
                list[pos] = u;
                umask[pos] = m;
            }
            n += __popc(b);
            tm |= __reduce_or_sync(0xffffffffu, m);
        }
        if (lane == 0) {
            meta[0] = n;
            meta[1] = static_cast<int>(tm);
        }
    }
    __syncthreads();
    const int nk = meta[0];
    const unsigned tmask = static_cast<unsigned>(meta[1]);
    // the listed units' rows of Wd_s move to L2 while their rows of Wu_s are read and used
    for (int k = threadIdx.x; k < nk; k += blockDim.x)
        bulk_prefetch_l2(Wd + static_cast<size_t>(u_base + list[k]) * d, static_cast<uint32_t>(d) * 2u);

    // up projection: one warp per listed unit, lanes on 16-byte chunks lane, lane + 32, ... of the
    // row, eight at a time
    const int chunks = d / 8;
    // h = a * u with a as the TwELL stores it (fp32 g, or g rounded to bf16)
    auto store_h = [&](int u, int r, float dot) {
        const float g = gs[u * NTOK + r];
        const float a = vals_f32 ? g : __bfloat162float(__float2bfloat16_rn(g));
        hs[u * NTOK + r] = a * dot;
    };
    if (chunks <= 32 * kDecodeChunks) {
        // the row fits one batch of chunks: load it once, then one token of the mask at a time
        for (int k = warp; k < nk; k += kSmallWarps) {
            const int u = list[k];
            const __nv_bfloat16* wr = Wu + static_cast<size_t>(u_base + u) * d;
            uint4 w[kDecodeChunks];
#pragma unroll
            for (int i = 0; i < kDecodeChunks; ++i) {
                const int c = lane + 32 * i;
                w[i] = c < chunks ? ldg_stream16(wr + c * 8) : make_uint4(0u, 0u, 0u, 0u);
            }
            for (unsigned m = umask[k]; m != 0u; m &= m - 1u) {
                const int r = __ffs(m) - 1;
                const uint8_t* xr = xs + r * L.G.x_stride;
                float v = 0.0f;
#pragma unroll
                for (int i = 0; i < kDecodeChunks; ++i) {
                    const int c = lane + 32 * i;
                    if (c < chunks) v += dot8(w[i], *reinterpret_cast<const uint4*>(xr + c * 16));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) store_h(u, r, v);
            }
        }
    } else {
        // wider rows: all keeping tokens' dots in one pass per batch of chunks
        for (int k = warp; k < nk; k += kSmallWarps) {
            const int u = list[k];
            const unsigned m = umask[k];
            const __nv_bfloat16* wr = Wu + static_cast<size_t>(u_base + u) * d;
            float s[NTOK];
#pragma unroll
            for (int r = 0; r < NTOK; ++r) s[r] = 0.0f;
            for (int c0 = lane; c0 < chunks; c0 += 32 * kDecodeChunks) {
                uint4 w[kDecodeChunks];
#pragma unroll
                for (int i = 0; i < kDecodeChunks; ++i) {
                    const int c = c0 + 32 * i;
                    w[i] = c < chunks ? ldg_stream16(wr + c * 8) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int r = 0; r < NTOK; ++r) {
                    if (!((m >> r) & 1u)) continue;
                    const uint8_t* xr = xs + r * L.G.x_stride;
#pragma unroll
                    for (int i = 0; i < kDecodeChunks; ++i) {
                        const int c = c0 + 32 * i;
                        if (c < chunks) s[r] += dot8(w[i], *reinterpret_cast<const uint4*>(xr + c * 16));
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < NTOK; ++r) {
                if (!((m >> r) & 1u)) continue;
                float v = s[r];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) store_h(u, r, v);
            }
        }
    }
    __syncthreads();

    // down projection: thread owns 4 columns at a time, for 8 tokens at a time; units in list order
    const size_t blk = blockIdx.x;
    for (int r0 = 0; r0 < NTOK; r0 += 8) {
        if (((tmask >> r0) & 0xffu) == 0u) continue;
        for (int c4 = threadIdx.x; c4 < d / 4; c4 += blockDim.x) {
            float acc[8][4];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.0f;
#pragma unroll 4
            for (int k = 0; k < nk; ++k) {
                const int u = list[k];
                const uint2 wv = __ldg(reinterpret_cast<const uint2*>(Wd + static_cast<size_t>(u_base + u) * d) + c4);
                const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv.x));
                const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv.y));
                const float* hu = hs + u * NTOK + r0;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const float h = hu[r];
                    acc[r][0] = fmaf(h, w01.x, acc[r][0]);
                    acc[r][1] = fmaf(h, w01.y, acc[r][1]);
                    acc[r][2] = fmaf(h, w23.x, acc[r][2]);
                    acc[r][3] = fmaf(h, w23.y, acc[r][3]);
                }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if (r0 + r < N && ((tmask >> (r0 + r)) & 1u))
                    reinterpret_cast<float4*>(part_y + (blk * N + r0 + r) * static_cast<size_t>(d))[c4] =
                        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
            }
        }
    }
    if (threadIdx.x < N) flags[blk * N + threadIdx.x] = (tmask >> threadIdx.x) & 1u;
    cluster.sync();  // the peer's g stays in place until both CTAs have read it
}

// y[r, 4c .. 4c+3] = the sum of token r's flagged partial rows. Block (column block, token): the
// flags are read once and the used CTAs listed in ascending order; thread (j, c) adds list entries
// j, j + 4, ... (loads independent of one another), and the four sums are added in the order
// 0 + 1 + 2 + 3: a fixed order, so y does not depend on scheduling.
constexpr int kReduceCols = 64;  // float4 columns per block
constexpr int kReduceWays = 4;   // list entries split over this many threads per column
__global__ void __launch_bounds__(kReduceCols * kReduceWays) decode_reduce_kernel(const float* __restrict__ part_y,
                                                                                  const int* __restrict__ flags,
                                                                                  int ncta, int N, int d,
                                                                                  __nv_bfloat16* __restrict__ y)
{
    extern __shared__ int s_list[];  // [ncta] used CTAs, then [kReduceWays * kReduceCols] float4 sums
    __shared__ int s_n;
    // launched as a programmatic dependent of decode_small_kernel: wait until that grid has finished
    // and its partial rows and flags are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int r = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp == 0) {
        int n = 0;
        for (int b0 = 0; b0 < ncta; b0 += 32) {
            const int b = b0 + lane;
            const bool used = b < ncta && flags[static_cast<size_t>(b) * N + r] != 0;
            const unsigned m = __ballot_sync(0xffffffffu, used);
            if (used) s_list[n + __popc(m & ((1u << lane) - 1u))] = b;
            n += __popc(m);
        }
        if (lane == 0) s_n = n;
    }
    __syncthreads();
    const int n = s_n;
    const int j = threadIdx.x / kReduceCols, cl = threadIdx.x % kReduceCols;
    const int c4 = blockIdx.x * kReduceCols + cl;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (c4 < d / 4) {
#pragma unroll 8
        for (int i = j; i < n; i += kReduceWays) {
            const float4 v =
                __ldg(reinterpret_cast<const float4*>(part_y + (static_cast<size_t>(s_list[i]) * N + r) * d) + c4);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
    }
    float4* s_acc = reinterpret_cast<float4*>(s_list + ((ncta + 3) & ~3));
    s_acc[j * kReduceCols + cl] = acc;
    __syncthreads();
    if (j == 0 && c4 < d / 4) {
#pragma unroll
        for (int w = 1; w < kReduceWays; ++w) {
            const float4 v = s_acc[w * kReduceCols + cl];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&lo);
        o.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(y + static_cast<size_t>(r) * d)[c4] = o;
    }
}

template <int NB, int T>
twell_status launch_decode(const __nv_bfloat16* x, const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                           const __nv_bfloat16* Wd, int N, int d, int f, int nt, const twell_packed* a,
                           __nv_bfloat16* y, void* ws, cudaStream_t s)
{
    const DecodeLayout L(NB, T, d);
    const DecodeWs W(N, d, f, T);
    auto kern = decode_small_kernel<NB, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total)) !=
        cudaSuccess)
        return TWELL_ERR_CUDA;
    int* flags = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + W.flags);
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + W.part);
    kern<<<2 * nt, 32 * kSmallWarps, L.total, s>>>(x, Wg, Wu, Wd, N, d, f, nt, a->dtype == TWELL_F32 ? 1 : 0, a->vals,
                                                   a->idx, a->cnt, part, flags);
    if (twell_host::launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    const int ncta = 2 * nt;
    const size_t rsmem = static_cast<size_t>((ncta + 3) & ~3) * 4 + kReduceWays * kReduceCols * 16;
    if (rsmem > 48 * 1024) return TWELL_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((d / 4 + kReduceCols - 1) / kReduceCols, N);
    cfg.blockDim = dim3(kReduceCols * kReduceWays);
    cfg.dynamicSmemBytes = rsmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_reduce_kernel, static_cast<const float*>(part), static_cast<const int*>(flags),
                           ncta, N, d, y) != cudaSuccess)
        return TWELL_ERR_CUDA;
    return twell_host::launch_status();
}

template <int NB>
twell_status run_decode(const __nv_bfloat16* x, const __nv_bfloat16* Wg, const __nv_bfloat16* Wu,
                        const __nv_bfloat16* Wd, int N, int d, int f, int T, int nt, const twell_packed* a,
                        __nv_bfloat16* y, void* ws, cudaStream_t s)
{
    switch (T) {
    case 64: return launch_decode<NB, 64>(x, Wg, Wu, Wd, N, d, f, nt, a, y, ws, s);
    case 128: return launch_decode<NB, 128>(x, Wg, Wu, Wd, N, d, f, nt, a, y, ws, s);
    case 256: return launch_decode<NB, 256>(x, Wg, Wu, Wd, N, d, f, nt, a, y, ws, s);
    default: return TWELL_ERR_UNSUPPORTED;
    }
}

}  // namespace
}  // namespace twell

size_t twell_host::decode_ws_bytes(int N, int d, int f, int T) { return twell::DecodeWs(N, d, f, T).total; }

using namespace twell_host;

extern "C" twell_status twell_ffn_decode(const void* x, const void* Wg_s, const void* Wu_s, const void* Wd_s,
                                         int32_t N, int32_t d, int32_t f, int32_t T, const twell_packed* a_out,
                                         void* y, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream)
{
    if (Wg_s == nullptr || Wu_s == nullptr || Wd_s == nullptr || a_out == nullptr || dev_status == nullptr)
        return TWELL_ERR_INVALID;
    if ((x == nullptr || y == nullptr) && N != 0) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0) return TWELL_ERR_INVALID;
    if (N > twell::kSmallMaxN || d % 64 != 0 || d > 4096 || (T != 64 && T != 128 && T != 256))
        return TWELL_ERR_UNSUPPORTED;
    if (!dtype_ok(a_out->dtype)) return TWELL_ERR_UNSUPPORTED;
    twell_status st = check_packed(a_out, N, f, T, a_out->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    if (ws == nullptr || ws_bytes < twell::DecodeWs(N, d, f, T).total) return TWELL_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(Wg_s) || !aligned16(Wu_s) || !aligned16(Wd_s) || !aligned16(y) ||
        !aligned16(ws))
        return TWELL_ERR_INVALID;
    using bf = __nv_bfloat16;
    const int nt = (f + T - 1) / T;
    const bf *xb = static_cast<const bf*>(x), *g = static_cast<const bf*>(Wg_s), *u = static_cast<const bf*>(Wu_s),
             *w = static_cast<const bf*>(Wd_s);
    bf* yb = static_cast<bf*>(y);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return N <= 8 ? twell::run_decode<1>(xb, g, u, w, N, d, f, T, nt, a_out, yb, ws, s)
                  : twell::run_decode<2>(xb, g, u, w, N, d, f, T, nt, a_out, yb, ws, s);
}
