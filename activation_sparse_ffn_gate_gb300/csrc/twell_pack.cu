// twell_pack.cu -- TwELL pack of a given gate matrix and TwELL unpack (test exports); per-column
// activity counts of a TwELL matrix and a row gather, the two steps of dead-column compaction.
//
// One warp per (token row, column tile): the lanes test 32 columns at a time, a warp ballot marks
// the kept entries (g > 0) and each kept lane finds its slot as the population count of the
// ballot bits below it -- the same ascending-order compaction the gate epilogue performs
// ([TG] "Вот тут и решает TwELL"; [TC] §2).
#include "twell_common.cuh"

namespace twell {

template <typename E, typename VO = E>
__global__ void pack_from_gate_kernel(const E* __restrict__ G, int N, int f, int T, int nt, VO* __restrict__ vals,
                                      uint8_t* __restrict__ idx, uint16_t* __restrict__ cnt)
{
    const int lane = threadIdx.x & 31;
    const long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= static_cast<long long>(N) * nt) return;
    const int r = static_cast<int>(w / nt), t = static_cast<int>(w % nt);
    const size_t slot = (static_cast<size_t>(r) * nt + t) * T;
    int c = 0;
    for (int ch = 0; ch < T; ch += 32) {
        const int k = ch + lane;
        const int j = t * T + k;
        E g{};
        bool keep = false;
        if (j < f) {
            g = G[static_cast<size_t>(r) * f + j];
            keep = Elem<E>::to_f(g) > 0.0f;
        }
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        const int pos = c + __popc(m & ((1u << lane) - 1u));
        if (keep) {
            vals[slot + pos] = static_cast<VO>(Elem<E>::to_f(g));
            idx[slot + pos] = static_cast<uint8_t>(k);
        }
        c += __popc(m);
    }
    if (lane == 0) cnt[static_cast<size_t>(r) * nt + t] = static_cast<uint16_t>(c);
}

template <typename E>
__global__ void unpack_kernel(const E* __restrict__ vals, const uint8_t* __restrict__ idx,
                              const uint16_t* __restrict__ cnt, int N, int f, int T, int nt, E* __restrict__ dense,
                              int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= static_cast<long long>(N) * nt) return;
    const int r = static_cast<int>(w / nt), t = static_cast<int>(w % nt);
    E* out = dense + static_cast<size_t>(r) * f;
    for (int k = lane; k < T; k += 32) {
        const int j = t * T + k;
        if (j < f) out[j] = Elem<E>::from_f(0.0f);
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
        if (j < f) out[j] = vals[slot + k];
        else report(status, TWELL_ERR_DEVICE_CHECK);
    }
}

// One warp per (token row, column tile): each kept entry adds one to its column's count. A count
// above the tile width or a column at or beyond n_cols is recorded and skipped.
__global__ void column_activity_kernel(const uint8_t* __restrict__ idx, const uint16_t* __restrict__ cnt, int N,
                                       int f, int T, int nt, int32_t* __restrict__ col_counts, int32_t* status)
{
    const int lane = threadIdx.x & 31;
    const long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= static_cast<long long>(N) * nt) return;
    const int t = static_cast<int>(w % nt);
    const int c = cnt[w];
    if (c > T) {
        if (lane == 0) report(status, TWELL_ERR_DEVICE_CHECK);
        return;
    }
    for (int q = lane; q < c; q += 32) {
        const int k = idx[w * T + q];
        const int j = t * T + k;
        if (k >= T || j >= f) {
            report(status, TWELL_ERR_DEVICE_CHECK);
            continue;
        }
        atomicAdd(&col_counts[j], 1);
    }
}

// total += the sum of the TwELL counts (its kept entries); a count above the tile width is
// recorded and counted as 0. Grid-stride over the counts, a warp sum, one atomic per warp.
__global__ void count_nonzeros_kernel(const uint16_t* __restrict__ cnt, long long n, int T,
                                      unsigned long long* __restrict__ total, int32_t* status)
{
    unsigned long long s = 0;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int c = cnt[i];
        if (c > T) report(status, TWELL_ERR_DEVICE_CHECK);
        else s += static_cast<unsigned long long>(c);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0 && s != 0) atomicAdd(total, s);
}

// dst[i, :] = src[rows[i], :] in 16-byte chunks; a row index outside [0, n_src) is recorded and
// its output row is zero.
__global__ void gather_rows_checked_kernel(const uint4* __restrict__ src, int n_src, const int32_t* __restrict__ rows,
                                           int n, int chunks, uint4* __restrict__ dst, int32_t* status)
{
    const long long total = static_cast<long long>(n) * chunks;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(e / chunks), q = static_cast<int>(e % chunks);
        const int r = rows[i];
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r >= 0 && r < n_src) v = src[static_cast<size_t>(r) * chunks + q];
        else if (q == 0) report(status, TWELL_ERR_DEVICE_CHECK);
        dst[e] = v;
    }
}

}  // namespace twell

using namespace twell_host;

static inline unsigned warp_blocks(long long warps, int per_block)
{
    return static_cast<unsigned>((warps + per_block - 1) / per_block);
}

extern "C" twell_status twell_pack_from_gate(const void* G, int32_t N, int32_t f, int32_t T, twell_dtype dtype,
                                             const twell_packed* out, int32_t* dev_status, void* stream)
{
    if (dev_status == nullptr || (G == nullptr && N != 0)) return TWELL_ERR_INVALID;
    if (N < 0 || f <= 0) return TWELL_ERR_INVALID;
    if (!dtype_ok(dtype)) return TWELL_ERR_UNSUPPORTED;
    twell_status st = check_packed(out, N, f, T, dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    if (!aligned16(G)) return TWELL_ERR_INVALID;
    const int nt = (f + T - 1) / T;
    const long long warps = static_cast<long long>(N) * nt;
    if (warps / 8 + 1 > 0x7fffffffLL) return TWELL_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == TWELL_BF16)
        twell::pack_from_gate_kernel<__nv_bfloat16><<<warp_blocks(warps, 8), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(G), N, f, T, nt, static_cast<__nv_bfloat16*>(out->vals), out->idx,
            out->cnt);
    else
        twell::pack_from_gate_kernel<float><<<warp_blocks(warps, 8), 256, 0, s>>>(
            static_cast<const float*>(G), N, f, T, nt, static_cast<float*>(out->vals), out->idx, out->cnt);
    return launch_status();
}

twell_status twell_host::pack_gate_widened(const void* G, int N, int f, const twell_packed* out, int32_t* status,
                                          cudaStream_t s)
{
    (void)status;
    if (out == nullptr || out->dtype != TWELL_F32) return TWELL_ERR_INVALID;
    const int T = out->tile, nt = (f + T - 1) / T;
    const long long warps = static_cast<long long>(N) * nt;
    if (N == 0) return TWELL_OK;
    twell::pack_from_gate_kernel<__nv_bfloat16, float><<<warp_blocks(warps, 8), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(G), N, f, T, nt, static_cast<float*>(out->vals), out->idx, out->cnt);
    return launch_status();
}

extern "C" twell_status twell_unpack(const twell_packed* a, void* dense_out, int32_t* dev_status, void* stream)
{
    if (a == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if (!dtype_ok(a->dtype)) return TWELL_ERR_UNSUPPORTED;
    const int N = a->n_rows, f = a->n_cols, T = a->tile;
    if (N < 0 || f <= 0 || (dense_out == nullptr && N != 0)) return TWELL_ERR_INVALID;
    twell_status st = check_packed(a, N, f, T, a->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    if (!aligned16(dense_out)) return TWELL_ERR_INVALID;
    const int nt = (f + T - 1) / T;
    const long long warps = static_cast<long long>(N) * nt;
    if (warps / 8 + 1 > 0x7fffffffLL) return TWELL_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (a->dtype == TWELL_BF16)
        twell::unpack_kernel<__nv_bfloat16><<<warp_blocks(warps, 8), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(a->vals), a->idx, a->cnt, N, f, T, nt,
            static_cast<__nv_bfloat16*>(dense_out), dev_status);
    else
        twell::unpack_kernel<float><<<warp_blocks(warps, 8), 256, 0, s>>>(static_cast<const float*>(a->vals), a->idx,
                                                                          a->cnt, N, f, T, nt,
                                                                          static_cast<float*>(dense_out), dev_status);
    return launch_status();
}

extern "C" twell_status twell_column_activity(const twell_packed* a, int32_t* col_counts, int32_t* dev_status,
                                              void* stream)
{
    if (a == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if (!dtype_ok(a->dtype)) return TWELL_ERR_UNSUPPORTED;
    const int N = a->n_rows, f = a->n_cols, T = a->tile;
    if (N < 0 || f <= 0 || col_counts == nullptr) return TWELL_ERR_INVALID;
    twell_status st = check_packed(a, N, f, T, a->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    const int nt = (f + T - 1) / T;
    const long long warps = static_cast<long long>(N) * nt;
    if (warps / 8 + 1 > 0x7fffffffLL) return TWELL_ERR_UNSUPPORTED;
    twell::column_activity_kernel<<<warp_blocks(warps, 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        a->idx, a->cnt, N, f, T, nt, col_counts, dev_status);
    return launch_status();
}

extern "C" twell_status twell_count_nonzeros(const twell_packed* a, unsigned long long* total, int32_t* dev_status,
                                             void* stream)
{
    if (a == nullptr || dev_status == nullptr || total == nullptr) return TWELL_ERR_INVALID;
    if (!dtype_ok(a->dtype)) return TWELL_ERR_UNSUPPORTED;
    const int N = a->n_rows, f = a->n_cols, T = a->tile;
    if (N < 0 || f <= 0) return TWELL_ERR_INVALID;
    twell_status st = check_packed(a, N, f, T, a->dtype);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    DevInfo di;
    if (dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    const long long n = static_cast<long long>(N) * ((f + T - 1) / T);
    const long long need = (n + 255) / 256;
    const int grid = static_cast<int>(need < 4ll * di.sm_count ? need : 4ll * di.sm_count);
    twell::count_nonzeros_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a->cnt, n, T, total, dev_status);
    return launch_status();
}

extern "C" twell_status twell_gather_rows(const void* src, int32_t n_src, const int32_t* rows, int32_t n, int32_t d,
                                          twell_dtype dtype, void* dst, int32_t* dev_status, void* stream)
{
    if (dev_status == nullptr || n_src < 0 || n < 0 || d <= 0) return TWELL_ERR_INVALID;
    if (!dtype_ok(dtype)) return TWELL_ERR_UNSUPPORTED;
    const int esz = dtype == TWELL_BF16 ? 2 : 4;
    if ((static_cast<long long>(d) * esz) % 16 != 0) return TWELL_ERR_INVALID;
    if (n == 0) return TWELL_OK;
    if (src == nullptr || rows == nullptr || dst == nullptr) return TWELL_ERR_INVALID;
    if (!aligned16(src) || !aligned16(dst)) return TWELL_ERR_INVALID;
    const int chunks = static_cast<int>(static_cast<long long>(d) * esz / 16);
    DevInfo di;
    if (dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    const long long total = static_cast<long long>(n) * chunks;
    long long blocks = (total + 255) / 256;
    if (blocks > 8LL * di.sm_count) blocks = 8LL * di.sm_count;
    twell::gather_rows_checked_kernel<<<static_cast<int>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(src), n_src, rows, n, chunks, static_cast<uint4*>(dst), dev_status);
    return launch_status();
}

// ------------------------------------------------------------------------------------------
// The bounded wait on its own (see twell_wait_probe in include/twell.h).

namespace twell {
namespace {
__global__ void wait_probe_kernel(int arrive, uint64_t limit_ns, int32_t* status)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    wait_bounded(&bar, 0u, nullptr, status, limit_ns);
}
}  // namespace
}  // namespace twell

extern "C" twell_status twell_wait_probe(int32_t arrive, int32_t limit_ms, int32_t* dev_status, void* stream)
{
    if (dev_status == nullptr || limit_ms < 1 || limit_ms > 10000) return TWELL_ERR_INVALID;
    twell::wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        arrive != 0, static_cast<uint64_t>(limit_ms) * 1000000ull, dev_status);
    return launch_status();
}
