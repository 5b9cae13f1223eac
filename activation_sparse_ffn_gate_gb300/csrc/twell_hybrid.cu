// twell_hybrid.cu -- hybrid sparse-block / dense-backup format for training: forward and backward.
//
// Each token row is routed by its number of kept gate activations nnz_r ([TG] "Обучение";
// [TC] §3): rows with nnz_r <= K are squeezed into one globally aligned sparse block of K slots
// (columns ascending, padded), rows with nnz_r > K go to a dense backup buffer in ascending row
// order. Light rows are computed by gathering rows of the weights (CUDA cores, no dense product);
// backup rows by dense tcgen05 GEMMs on the gathered rows ([TC] §3: tensor cores take the heavy
// rows, custom sparse kernels the light ones). The backward pass of the light rows has no
// product of two dense matrices ([TG] "Обучение"): the weight gradients of the sparse entries
// are formed per hidden unit after a column-wise regrouping of the entries.
//
// Loss whose gradients are computed: L = <y, dy> + lambda * mean|h| over all N*f entries of h
// ([AIM] ¶4; [PUL] ¶4: L1 coefficient 2e-5 on the hidden activations).
#include <mutex>
#include <type_traits>

#include "twell_gemm.cuh"
#include "twell_light.cuh"

namespace twell {

constexpr int kHybTile = 128;   // TwELL tile of the gate epilogue inside the hybrid path
constexpr int kRouteRows = 32;  // rows per routing block (two per warp: short dependent-load chains)
constexpr int kRowBatch = 8;    // nonzeros per batch in the light-row kernels
constexpr int kMaxK = 65534;    // largest capacity K (counts are uint16, 0xFFFF marks a backup row)
constexpr int kBackupSplits = 4; // K ranges of the backup rows' y and dx products (few rows, long K)

// ------------------------------------------------------------------------------------------
// Workspace layout (offsets in bytes from ws, each 256-byte aligned)

struct HybridWs {
    int nt, nblk, f_pad;
    size_t capr;  // backup rows rounded up to a 64-row k-block (zero-padded rows)
    // routing / forward
    size_t tw_vals, tw_idx, tw_cnt, blk, l1acc, tick, route_total, x_b, h_b, y_part, fwd_total;
    // backward
    size_t ent, btick, ccount, coff, ccur, rec, dy_b, dh_b, dug, dx_part, bwd_total;
    static size_t al(size_t v) { return (v + 255) & ~size_t(255); }
    HybridWs(int N, int d, int f, int K, int cap)
    {
        nt = (f + kHybTile - 1) / kHybTile;
        nblk = (N + kRouteRows - 1) / kRouteRows;
        f_pad = (f + 63) / 64 * 64;
        capr = static_cast<size_t>((cap + 63) / 64 * 64);
        size_t o = 0;
        tw_vals = o;
        o = al(o + static_cast<size_t>(N) * nt * kHybTile * 4);
        tw_idx = o;
        o = al(o + static_cast<size_t>(N) * nt * kHybTile);
        tw_cnt = o;
        o = al(o + static_cast<size_t>(N) * nt * 2);
        blk = o;
        o = al(o + static_cast<size_t>(nblk) * 4);
        l1acc = o;
        o = al(o + 16);
        tick = o;  // row counter of the light-row kernel
        o = al(o + 16);
        x_b = o;
        o = al(o + capr * d * 2);
        route_total = o;
        h_b = o;
        o = al(o + capr * 2 * f_pad * 2);  // [h_hi | h_lo] bf16
        y_part = o;
        o = al(o + kBackupSplits * capr * d * 4);  // fp32 partial y of the backup rows, per K range
        fwd_total = o;
        o = 0;
        ent = o;
        o = al(o + static_cast<size_t>(N) * K * 12);
        btick = o;
        o = al(o + 16);
        ccount = o;
        o = al(o + static_cast<size_t>(f) * 4);
        coff = o;
        o = al(o + static_cast<size_t>(f + 1) * 4);
        ccur = o;
        o = al(o + static_cast<size_t>(f) * 4);
        rec = o;  // records of the light entries and of the backup rows' kept entries
        o = al(o + (static_cast<size_t>(N) * K + static_cast<size_t>(cap) * f) * 16);
        dy_b = o;
        o = al(o + capr * d * 2);
        dh_b = o;
        o = al(o + capr * f_pad * 4);
        dug = o;
        o = al(o + capr * 4 * f_pad * 2);  // [du_hi | dg_hi | du_lo | dg_lo] bf16
        dx_part = o;
        o = al(o + kBackupSplits * capr * d * 4);  // fp32 partial dx of the backup rows, per K range
        bwd_total = o;
    }
};

// ------------------------------------------------------------------------------------------
// Routing

constexpr int kRouteWarps = 16;                          // warps of a routing block (two rows each)
constexpr int kRouteMaxTiles = (65535 + kHybTile - 1) / kHybTile;  // d_ff <= 65535

// Per row (one warp): nnz from the TwELL counts, scanned into per-tile offsets in shared memory;
// a light row (nnz <= K) is written into the sparse block in ascending column order, one entry per
// lane at a time (its tile found by binary search over the offsets), and padded; a heavy row is
// marked 0xFFFF. Per block: number of heavy rows.
__global__ void __launch_bounds__(32 * kRouteWarps) route_rows_kernel(
    const float* __restrict__ vals, const uint8_t* __restrict__ idx, const uint16_t* __restrict__ cnt, int N, int f,
    int nt, int K, float* __restrict__ ha, uint16_t* __restrict__ hcol, uint16_t* __restrict__ hcnt,
    int* __restrict__ blk, double* l1acc, int32_t* status)
{
    pdl_begin();
    __shared__ int s_pref[kRouteWarps][kRouteMaxTiles + 1];
    __shared__ int s_heavy;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int* pref = s_pref[warp];
    if (threadIdx.x == 0) s_heavy = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0 && l1acc != nullptr) *l1acc = 0.0;
    __syncthreads();
    const int r0 = blockIdx.x * kRouteRows;
    for (int rr = warp; rr < kRouteRows; rr += nw) {
        const int r = r0 + rr;
        if (r >= N) break;
        int run = 0;
        for (int t0 = 0; t0 < nt; t0 += 32) {
            const int t = t0 + lane;
            int c = t < nt ? cnt[static_cast<size_t>(r) * nt + t] : 0;
            if (c > kHybTile) {
                report(status, TWELL_ERR_DEVICE_CHECK);
                c = 0;
            }
            int inc = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += u;
            }
            if (t < nt) pref[t] = run + inc - c;
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) pref[nt] = run;
        __syncwarp();
        if (run <= K) {
            for (int p = lane; p < run; p += 32) {
                int lo = 0, hi = nt;  // the last tile with pref[tile] <= p holds entry p
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (pref[mid] <= p) lo = mid;
                    else hi = mid;
                }
                const size_t e = (static_cast<size_t>(r) * nt + lo) * kHybTile + (p - pref[lo]);
                ha[static_cast<size_t>(r) * K + p] = vals[e];
                hcol[static_cast<size_t>(r) * K + p] = static_cast<uint16_t>(lo * kHybTile + idx[e]);
            }
            for (int k = run + lane; k < K; k += 32) {
                ha[static_cast<size_t>(r) * K + k] = 0.0f;
                hcol[static_cast<size_t>(r) * K + k] = 0;
            }
            if (lane == 0) hcnt[r] = static_cast<uint16_t>(run);
        } else if (lane == 0) {
            hcnt[r] = 0xFFFF;
            atomicAdd(&s_heavy, 1);
        }
        __syncwarp();  // every lane is done with the offsets before the next row overwrites them
    }
    __syncthreads();
    if (threadIdx.x == 0) blk[blockIdx.x] = s_heavy;
}

// Backup slots in ascending row order: block b's heavy rows start after all heavy rows of blocks
// < b (their counts are summed directly, no inter-CTA waiting). For each heavy row with a slot
// below cap (one warp per row): backup_rows[slot] = r, A_b[slot] = its dense ReLU(g) row (fp32),
// x_b[slot] = x_r.
__global__ void route_backup_kernel(const float* __restrict__ vals, const uint8_t* __restrict__ idx,
                                    const uint16_t* __restrict__ cnt, const uint16_t* __restrict__ hcnt,
                                    const int* __restrict__ blk, int nblk, int N, int f, int nt, int cap,
                                    const __nv_bfloat16* __restrict__ x, int d, int32_t* __restrict__ brows,
                                    int32_t* __restrict__ n_backup, float* __restrict__ A_b,
                                    __nv_bfloat16* __restrict__ x_b, int32_t* status)
{
    pdl_begin();
    __shared__ int s_off, s_total, s_rank[kRouteRows];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    if (tid < 32) {
        int before = 0, total = 0;
        for (int b = tid; b < nblk; b += 32) {
            const int c = blk[b];
            total += c;
            if (b < blockIdx.x) before += c;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, o);
            total += __shfl_xor_sync(0xffffffffu, total, o);
        }
        if (tid == 0) {
            s_off = before;
            s_total = total;
            if (blockIdx.x == 0) {
                *n_backup = total;
                if (total > cap) report(status, TWELL_ERR_BACKUP_FULL);
            }
        }
        // ranks of this block's heavy rows, in row order
        int run = 0;
        for (int rr0 = 0; rr0 < kRouteRows; rr0 += 32) {
            const int r = blockIdx.x * kRouteRows + rr0 + tid;
            const bool heavy = r < N && hcnt[r] == 0xFFFF;
            const unsigned m = __ballot_sync(0xffffffffu, heavy);
            s_rank[rr0 + tid] = heavy ? run + __popc(m & ((1u << tid) - 1u)) : -1;
            run += __popc(m);
        }
    }
    __syncthreads();
    int seen = 0;  // heavy rows of this block met so far: the warp takes every nw-th
    for (int rr = 0; rr < kRouteRows; ++rr) {
        const int rank = s_rank[rr];
        if (rank < 0) continue;
        if (seen++ % nw != warp) continue;
        const int slot = s_off + rank;
        if (slot >= cap) continue;
        const int r = blockIdx.x * kRouteRows + rr;
        if (lane == 0) brows[slot] = r;
        float* arow = A_b + static_cast<size_t>(slot) * f;
        if ((f & 3) == 0 && (reinterpret_cast<uintptr_t>(A_b) & 15) == 0) {  // rows 16-byte aligned
            float4* a4 = reinterpret_cast<float4*>(arow);
            for (int j = lane; j < f / 4; j += 32) a4[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        } else {
            for (int j = lane; j < f; j += 32) arow[j] = 0.0f;
        }
        __syncwarp();  // zeros before the kept values, across lanes
        for (int t = lane; t < nt; t += 32) {
            const int c = cnt[static_cast<size_t>(r) * nt + t];
            const size_t sb = (static_cast<size_t>(r) * nt + t) * kHybTile;
            for (int k = 0; k < c && k < kHybTile; ++k) {
                const int j = t * kHybTile + idx[sb + k];
                if (j < f) arow[j] = vals[sb + k];
            }
        }
        if (x != nullptr) {
            const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(r) * d);
            uint4* dst = reinterpret_cast<uint4*>(x_b + static_cast<size_t>(slot) * d);
            for (int q = lane; q < d / 8; q += 32) dst[q] = src[q];
        }
    }
    // zero x_b rows of the partly used last 64-row block (k padding of the backward GEMMs)
    if (blockIdx.x == 0 && x != nullptr) {
        const int nb = min(s_total, cap);
        const int pad_end = min((nb + 63) / 64 * 64, (cap + 63) / 64 * 64);
        for (size_t e = static_cast<size_t>(nb) * d / 8 + tid; e < static_cast<size_t>(pad_end) * d / 8; e += blockDim.x)
            reinterpret_cast<uint4*>(x_b)[e] = make_uint4(0, 0, 0, 0);
    }
}

// ------------------------------------------------------------------------------------------
// Light rows: forward and backward (one CTA per row, one thread per 16-byte chunk of d_model)

__device__ __forceinline__ void bf8(const uint4& v, float (&o)[8])
{
    unpack16(v, o, static_cast<__nv_bfloat16*>(nullptr));
}

// Block-wide sums of kRowBatch per-thread partials; every thread gets all totals.
__device__ __forceinline__ void block_sum8(float (&p)[kRowBatch], float (*s_red)[kRowBatch], int lane, int warp,
                                           int nw, float (&out)[kRowBatch])
{
#pragma unroll
    for (int k = 0; k < kRowBatch; ++k)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) p[k] += __shfl_xor_sync(0xffffffffu, p[k], o);
    if (lane == 0)
#pragma unroll
        for (int k = 0; k < kRowBatch; ++k) s_red[warp][k] = p[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRowBatch; ++k) {
        float s = 0.0f;
        for (int w = 0; w < nw; ++w) s += s_red[w][k];
        out[k] = s;
    }
    __syncthreads();
}

// y_r and u at the kept entries of light rows; sum |h| into l1acc.
__global__ void __launch_bounds__(512) hybrid_light_fwd_kernel(const __nv_bfloat16* __restrict__ x,
                                                               const __nv_bfloat16* __restrict__ Wu,
                                                               const __nv_bfloat16* __restrict__ Wd, int N, int d,
                                                               int f, int K, const float* __restrict__ ha,
                                                               const uint16_t* __restrict__ hcol,
                                                               const uint16_t* __restrict__ hcnt, float* __restrict__ hu,
                                                               __nv_bfloat16* __restrict__ y, double* l1acc,
                                                               int32_t* status)
{
    pdl_begin();
    __shared__ float s_red[16][kRowBatch];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int q = tid, nchunks = d / 8;
    float l1 = 0.0f;
    for (int r = blockIdx.x; r < N; r += gridDim.x) {
        const int n = hcnt[r];
        if (n == 0xFFFF) continue;  // backup row: the dense path writes y_r
        if (n > K) {
            report(status, TWELL_ERR_DEVICE_CHECK);
            continue;
        }
        float xv[8], acc[8];
        {
            const uint4 xr = q < nchunks ? *reinterpret_cast<const uint4*>(x + static_cast<size_t>(r) * d + q * 8)
                                         : make_uint4(0, 0, 0, 0);
            bf8(xr, xv);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
        for (int b = 0; b < n; b += kRowBatch) {
            const int nb = min(kRowBatch, n - b);
            uint4 wu[kRowBatch], wd[kRowBatch];
            float av[kRowBatch];
#pragma unroll
            for (int k = 0; k < kRowBatch; ++k) {
                const bool live = k < nb;
                int j = live ? hcol[static_cast<size_t>(r) * K + b + k] : 0;
                if (j >= f) {
                    report(status, TWELL_ERR_DEVICE_CHECK);
                    j = 0;
                }
                av[k] = live ? ha[static_cast<size_t>(r) * K + b + k] : 0.0f;
                const size_t off = static_cast<size_t>(j) * d + q * 8;
                wu[k] = (live && q < nchunks) ? ldg_stream16(Wu + off) : make_uint4(0, 0, 0, 0);
                wd[k] = (live && q < nchunks) ? ldg_stream16(Wd + off) : make_uint4(0, 0, 0, 0);
            }
            float p[kRowBatch], u[kRowBatch];
#pragma unroll
            for (int k = 0; k < kRowBatch; ++k) {
                float w[8];
                bf8(wu[k], w);
                float s = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(xv[e], w[e], s);
                p[k] = s;
            }
            block_sum8(p, s_red, lane, warp, nw, u);
#pragma unroll
            for (int k = 0; k < kRowBatch; ++k) {
                if (k >= nb) continue;
                const float h = av[k] * u[k];
                if (tid == 0) {
                    hu[static_cast<size_t>(r) * K + b + k] = u[k];
                    l1 += fabsf(h);
                }
                float w[8];
                bf8(wd[k], w);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(h, w[e], acc[e]);
            }
        }
        // padded slots of u hold 0
        for (int k = n + tid; k < K; k += blockDim.x) hu[static_cast<size_t>(r) * K + k] = 0.0f;
        if (q < nchunks)
            *reinterpret_cast<uint4*>(y + static_cast<size_t>(r) * d + q * 8) =
                pack16(acc, static_cast<__nv_bfloat16*>(nullptr));
    }
    if (tid == 0 && l1 != 0.0f) atomicAdd(l1acc, static_cast<double>(l1));
}

// Backward of light rows: dh, du, dg per kept entry (kept in `ent` as {h, du, dg}); dx_r.
__global__ void __launch_bounds__(512) hybrid_light_bwd_kernel(const __nv_bfloat16* __restrict__ dy,
                                                               const __nv_bfloat16* __restrict__ Wg,
                                                               const __nv_bfloat16* __restrict__ Wu,
                                                               const __nv_bfloat16* __restrict__ Wd, int N, int d,
                                                               int f, int K, const float* __restrict__ ha,
                                                               const float* __restrict__ hu,
                                                               const uint16_t* __restrict__ hcol,
                                                               const uint16_t* __restrict__ hcnt, float l1_scale,
                                                               float* __restrict__ ent, float* __restrict__ dx,
                                                               int32_t* status)
{
    pdl_begin();
    __shared__ float s_red[16][kRowBatch];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int q = tid, nchunks = d / 8;
    for (int r = blockIdx.x; r < N; r += gridDim.x) {
        const int n = hcnt[r];
        if (n == 0xFFFF) continue;
        if (n > K) {
            report(status, TWELL_ERR_DEVICE_CHECK);
            continue;
        }
        float dyv[8], acc[8];
        {
            const uint4 v = q < nchunks ? *reinterpret_cast<const uint4*>(dy + static_cast<size_t>(r) * d + q * 8)
                                        : make_uint4(0, 0, 0, 0);
            bf8(v, dyv);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
        for (int b = 0; b < n; b += kRowBatch) {
            const int nb = min(kRowBatch, n - b);
            uint4 wd[kRowBatch];
            int jj[kRowBatch];
#pragma unroll
            for (int k = 0; k < kRowBatch; ++k) {
                const bool live = k < nb;
                int j = live ? hcol[static_cast<size_t>(r) * K + b + k] : 0;
                if (j >= f) {
                    report(status, TWELL_ERR_DEVICE_CHECK);
                    j = 0;
                }
                jj[k] = j;
                wd[k] = (live && q < nchunks) ? ldg_stream16(Wd + static_cast<size_t>(j) * d + q * 8)
                                              : make_uint4(0, 0, 0, 0);
            }
            float p[kRowBatch], dh[kRowBatch];
#pragma unroll
            for (int k = 0; k < kRowBatch; ++k) {
                float w[8];
                bf8(wd[k], w);
                float s = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(dyv[e], w[e], s);
                p[k] = s;
            }
            block_sum8(p, s_red, lane, warp, nw, dh);
#pragma unroll
            for (int k = 0; k < kRowBatch; ++k) {
                if (k >= nb) continue;
                const size_t e0 = static_cast<size_t>(r) * K + b + k;
                const float av = ha[e0], uv = hu[e0];
                const float h = av * uv;
                const float sg = h > 0.0f ? 1.0f : (h < 0.0f ? -1.0f : 0.0f);
                const float g = dh[k] + l1_scale * sg;
                const float du = g * av, dg = g * uv;  // a > 0 at every kept entry
                if (tid == 0) {
                    ent[e0 * 3 + 0] = h;
                    ent[e0 * 3 + 1] = du;
                    ent[e0 * 3 + 2] = dg;
                }
                if (q < nchunks) {
                    const size_t off = static_cast<size_t>(jj[k]) * d + q * 8;
                    float wu[8], wg[8];
                    bf8(ldg_stream16(Wu + off), wu);
                    bf8(ldg_stream16(Wg + off), wg);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmaf(du, wu[e], fmaf(dg, wg[e], acc[e]));
                }
            }
        }
        if (q < nchunks) {
            float* o = dx + static_cast<size_t>(r) * d + q * 8;
            *reinterpret_cast<float4*>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4*>(o + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
}

// ------------------------------------------------------------------------------------------
// Column-wise regrouping of the light entries and the sparse weight gradients

__global__ void fill_i32_kernel(int* p, int n, int v)
{
    pdl_begin();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = v;
}

__global__ void col_hist_kernel(const uint16_t* __restrict__ hcol, const uint16_t* __restrict__ hcnt, int N, int K,
                                int f, int* __restrict__ ccount)
{
    pdl_begin();
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < static_cast<long long>(N) * K;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(e / K), k = static_cast<int>(e % K);
        const int n = hcnt[r];
        if (n == 0xFFFF || k >= n) continue;
        const int j = hcol[e];
        if (j < f) atomicAdd(&ccount[j], 1);
    }
}

// Exclusive scan of the f column counts (one CTA): coff[0..f], and a copy into the cursors.
__global__ void col_scan_kernel(const int* __restrict__ ccount, int f, int* __restrict__ coff, int* __restrict__ ccur)
{
    pdl_begin();
    __shared__ int s_w[32];
    __shared__ int s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0) s_carry = 0;
    __syncthreads();
    for (int base = 0; base < f; base += blockDim.x) {
        const int i = base + tid;
        const int c = i < f ? ccount[i] : 0;
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        if (lane == 31) s_w[warp] = inc;
        __syncthreads();
        int before = s_carry;
        for (int w = 0; w < warp; ++w) before += s_w[w];
        if (i < f) {
            coff[i] = before + inc - c;
            ccur[i] = before + inc - c;
        }
        __syncthreads();
        if (tid == 0) {
            int tot = 0;
            for (int w = 0; w < nw; ++w) tot += s_w[w];
            s_carry += tot;
        }
        __syncthreads();
    }
    if (tid == 0) coff[f] = s_carry;
}

struct EntRec {
    int row;
    float h, du, dg;
};

__global__ void col_scatter_kernel(const uint16_t* __restrict__ hcol, const uint16_t* __restrict__ hcnt, int N, int K,
                                   int f, const float* __restrict__ ent, int* __restrict__ ccur, EntRec* __restrict__ rec)
{
    pdl_begin();
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < static_cast<long long>(N) * K;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(e / K), k = static_cast<int>(e % K);
        const int n = hcnt[r];
        if (n == 0xFFFF || k >= n) continue;
        const int j = hcol[e];
        if (j >= f) continue;
        const int pos = atomicAdd(&ccur[j], 1);
        rec[pos] = EntRec{r, ent[e * 3], ent[e * 3 + 1], ent[e * 3 + 2]};
    }
}

// Columns with more than this many records are sorted in global memory by col_sort_kernel, the
// others in shared memory by col_dw_kernel.
constexpr int kDwSmemRecs = 512;

// Sort each long column's records by row (an insertion sort per column), so the per-column sums
// below run in a fixed order whatever order the scatter's atomics produced.
__global__ void col_sort_kernel(const int* __restrict__ coff, int f, EntRec* __restrict__ rec)
{
    pdl_begin();
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < f; j += gridDim.x * blockDim.x) {
        const int s = coff[j], e = coff[j + 1];
        if (e - s <= kDwSmemRecs) continue;
        for (int i = s + 1; i < e; ++i) {
            const EntRec v = rec[i];
            int k = i - 1;
            while (k >= s && rec[k].row > v.row) {
                rec[k + 1] = rec[k];
                --k;
            }
            rec[k + 1] = v;
        }
    }
}

// Weight gradients of the light entries, per hidden unit j over the records of column j in
// ascending row order (one CTA per hidden unit, one thread per 8 elements of d_model); overwrites
// dW. Two passes, so that the rows one pass gathers fit in L2 (x and dy together are twice its
// size at the 2B-like training shapes): PASS 0 dWg_s[j] = sum dg x_r and dWu_s[j] = sum du x_r,
// PASS 1 dWd_s[j] = sum h dy_r; the gathered rows are loaded with an evict-last L2 policy. A column
// of at most kDwSmemRecs records is ranked by row in shared memory (rows are distinct within a
// column); longer ones were sorted in place by col_sort_kernel. Records are taken four at a time
// so that each thread has four 16-byte loads in flight.
template <int PASS>
__global__ void __launch_bounds__(512) col_dw_kernel(const int* __restrict__ coff, const EntRec* __restrict__ rec,
                                                     int f, int d, const __nv_bfloat16* __restrict__ v,
                                                     float* __restrict__ dWa, float* __restrict__ dWb)
{
    pdl_begin();
    __shared__ EntRec s_in[kDwSmemRecs], s_out[kDwSmemRecs];
    const int q = threadIdx.x, nchunks = d / 8;
    const uint64_t pol = policy_evict_last();
    for (int j = blockIdx.x; j < f; j += gridDim.x) {
        const int s = coff[j], m = coff[j + 1] - s;
        const bool smem = m <= kDwSmemRecs;
        __syncthreads();  // the previous column's records are no longer read
        if (smem) {
            for (int i = q; i < m; i += blockDim.x) s_in[i] = rec[s + i];
            __syncthreads();
            for (int i = q; i < m; i += blockDim.x) {
                const int r = s_in[i].row;
                int rank = 0;
                for (int k = 0; k < m; ++k) rank += s_in[k].row < r ? 1 : 0;
                s_out[rank] = s_in[i];
            }
            __syncthreads();
        }
        const EntRec* R = smem ? s_out : rec + s;
        float aa[8] = {}, ab[8] = {};
        if (q < nchunks) {
            auto step = [&](const EntRec& rc, const uint4& vr) {
                float vv[8];
                bf8(vr, vv);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (PASS == 0) {
                        aa[t] = fmaf(rc.dg, vv[t], aa[t]);
                        ab[t] = fmaf(rc.du, vv[t], ab[t]);
                    } else {
                        aa[t] = fmaf(rc.h, vv[t], aa[t]);
                    }
                }
            };
            int i = 0;
            for (; i + 4 <= m; i += 4) {
                EntRec rc[4];
                uint4 vr[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    rc[k] = R[i + k];
                    vr[k] = ldg_l2hint16(v + static_cast<size_t>(rc[k].row) * d + q * 8, pol);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) step(rc[k], vr[k]);
            }
            for (; i < m; ++i) {
                const EntRec rc = R[i];
                step(rc, ldg_l2hint16(v + static_cast<size_t>(rc.row) * d + q * 8, pol));
            }
            const size_t o = static_cast<size_t>(j) * d + q * 8;
            *reinterpret_cast<float4*>(dWa + o) = make_float4(aa[0], aa[1], aa[2], aa[3]);
            *reinterpret_cast<float4*>(dWa + o + 4) = make_float4(aa[4], aa[5], aa[6], aa[7]);
            if (PASS == 0) {
                *reinterpret_cast<float4*>(dWb + o) = make_float4(ab[0], ab[1], ab[2], ab[3]);
                *reinterpret_cast<float4*>(dWb + o + 4) = make_float4(ab[4], ab[5], ab[6], ab[7]);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// Backup rows: elementwise steps around the dense GEMMs

// Split of an fp32 value into two bf16 terms, hi = bf16(v) and lo = bf16(v - hi): hi + lo keeps
// about 16 significant bits, so a GEMM over [hi | lo] against [B ; B] is accurate to ~2^-17.
__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo)
{
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// h = a * u for the backup rows (fp32 context), as [h_hi | h_lo] (bf16, row pitch 2 f_pad) for the
// y_b GEMM; sum |h| into l1acc. Pad columns [f, f_pad) hold 0.
__global__ void backup_h_kernel(const float* __restrict__ A_b, const float* __restrict__ U_b,
                                const int32_t* __restrict__ n_backup, int cap, int f, int f_pad,
                                __nv_bfloat16* __restrict__ H, double* l1acc)
{
    pdl_begin();
    const int nb = min(*n_backup, cap);
    float l1 = 0.0f;
    const long long total = static_cast<long long>(nb) * f_pad;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(e / f_pad), j = static_cast<int>(e % f_pad);
        float h = 0.0f;
        if (j < f) {
            const size_t s = static_cast<size_t>(i) * f + j;
            h = A_b[s] * U_b[s];
        }
        l1 += fabsf(h);
        __nv_bfloat16 hi, lo;
        split_bf16(h, hi, lo);
        H[static_cast<size_t>(i) * 2 * f_pad + j] = hi;
        H[static_cast<size_t>(i) * 2 * f_pad + f_pad + j] = lo;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    if ((threadIdx.x & 31) == 0 && l1 != 0.0f) atomicAdd(l1acc, static_cast<double>(l1));
}

// out[rowmap[m]] = the sum of part[s][m] over s = 0 .. splits-1 in that order, for m < min(*n, cap)
// (bf16 or fp32 rows of d elements; part: splits blocks of `stride` elements, row pitch d).
template <typename O>
__global__ void reduce_rows_kernel(const float* __restrict__ part, int splits, long long stride,
                                   const int32_t* __restrict__ n_dyn, int cap, int d, const int32_t* __restrict__ rowmap,
                                   O* __restrict__ out)
{
    pdl_begin();
    const int nb = min(*n_dyn, cap);
    const int q4 = d / 4;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < static_cast<long long>(nb) * q4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int m = static_cast<int>(i / q4), c = static_cast<int>(i % q4) * 4;
        float4 acc = *reinterpret_cast<const float4*>(part + static_cast<size_t>(m) * d + c);
        for (int sp = 1; sp < splits; ++sp) {
            const float4 v = *reinterpret_cast<const float4*>(part + sp * stride + static_cast<size_t>(m) * d + c);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        O* o = out + static_cast<size_t>(rowmap[m]) * d + c;
        if constexpr (std::is_same<O, float>::value) {
            *reinterpret_cast<float4*>(o) = acc;
        } else {
            o[0] = __float2bfloat16_rn(acc.x);
            o[1] = __float2bfloat16_rn(acc.y);
            o[2] = __float2bfloat16_rn(acc.z);
            o[3] = __float2bfloat16_rn(acc.w);
        }
    }
}

__global__ void l1_finalize_kernel(const double* l1acc, float scale, float* l1)
{
    pdl_begin();
    *l1 = static_cast<float>(*l1acc * static_cast<double>(scale));
}

// Gather rows: out[i] = src[rows[i]] for i < min(n, cap); rows [nb, ceil64(nb)) are zeroed.
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ src, const int32_t* __restrict__ rows,
                                   const int32_t* __restrict__ n_backup, int cap, int d,
                                   __nv_bfloat16* __restrict__ out)
{
    pdl_begin();
    const int nb = min(*n_backup, cap);
    const int pad_end = min((nb + 63) / 64 * 64, (cap + 63) / 64 * 64);
    const int nq = d / 8;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
         e < static_cast<long long>(pad_end) * nq; e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(e / nq), q = static_cast<int>(e % nq);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (i < nb) v = reinterpret_cast<const uint4*>(src + static_cast<size_t>(rows[i]) * d)[q];
        reinterpret_cast<uint4*>(out + static_cast<size_t>(i) * d)[q] = v;
    }
}

// Backup-row gradients at every column: dh = dH + lambda sgn(h)/(N f); du = dh a; dg = dh u [a>0].
// Writes DUG = [du_hi | dg_hi | du_lo | dg_lo] (bf16, row pitch 4 f_pad; the dx GEMM runs over all
// four against [Wu ; Wg ; Wu ; Wg]); rows [nb, ceil64(nb)) and pad columns are zero. Every kept
// entry (a > 0) of a backup row also becomes a column record {row, h, du, dg} for the per-unit
// weight gradients (its slot from the column cursor), as the light rows' entries do: a backup row
// keeps a few hundred of the d_ff units, so its weight gradients are sparse too.
__global__ void backup_grad_kernel(const float* __restrict__ A_b, const float* __restrict__ U_b,
                                   const float* __restrict__ dH, const int32_t* __restrict__ n_backup, int cap, int f,
                                   int f_pad, float l1_scale, const int32_t* __restrict__ brows, int* __restrict__ ccur,
                                   EntRec* __restrict__ rec, __nv_bfloat16* __restrict__ DUG)
{
    pdl_begin();
    const int nb = min(*n_backup, cap);
    const int rows = min((nb + 63) / 64 * 64, (cap + 63) / 64 * 64);
    const long long total = static_cast<long long>(rows) * f_pad;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(e / f_pad), j = static_cast<int>(e % f_pad);
        float du = 0.0f, dg = 0.0f, h = 0.0f;
        if (i < nb && j < f) {
            const size_t s = static_cast<size_t>(i) * f + j;
            const float a = A_b[s], u = U_b[s];
            h = a * u;
            const float sg = h > 0.0f ? 1.0f : (h < 0.0f ? -1.0f : 0.0f);
            const float g = dH[static_cast<size_t>(i) * f_pad + j] + l1_scale * sg;
            du = g * a;
            dg = a > 0.0f ? g * u : 0.0f;
            if (a > 0.0f) rec[atomicAdd(&ccur[j], 1)] = EntRec{brows[i], h, du, dg};
        }
        __nv_bfloat16 du_hi, du_lo, dg_hi, dg_lo;
        split_bf16(du, du_hi, du_lo);
        split_bf16(dg, dg_hi, dg_lo);
        __nv_bfloat16* row = DUG + static_cast<size_t>(i) * 4 * f_pad;
        row[j] = du_hi;
        row[f_pad + j] = dg_hi;
        row[2 * f_pad + j] = du_lo;
        row[3 * f_pad + j] = dg_lo;
    }
}

// Kept entries (a > 0) of the backup rows, per column: ccount[j] += #{i < min(nb, cap): A_b[i, j] > 0}.
__global__ void col_hist_backup_kernel(const float* __restrict__ A_b, const int32_t* __restrict__ n_backup, int cap,
                                       int f, int* __restrict__ ccount)
{
    pdl_begin();
    const int nb = min(*n_backup, cap);
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < static_cast<long long>(nb) * f;
         e += static_cast<long long>(gridDim.x) * blockDim.x)
        if (A_b[e] > 0.0f) atomicAdd(&ccount[e % f], 1);
}

}  // namespace twell

// ==========================================================================================
// C ABI

using namespace twell_host;
using bf = __nv_bfloat16;

namespace {

twell_status check_hybrid(const twell_hybrid* c, int N, int f, int K)
{
    if (c == nullptr) return TWELL_ERR_INVALID;
    if (c->n_rows != N || c->n_cols != f || c->K != K || c->backup_cap < 0) return TWELL_ERR_INVALID;
    if (c->dtype != TWELL_BF16) return TWELL_ERR_UNSUPPORTED;
    if (N == 0) return TWELL_OK;
    if (c->cnt == nullptr || c->n_backup == nullptr || c->dev_status == nullptr) return TWELL_ERR_INVALID;
    if (K > 0 && (c->a == nullptr || c->u == nullptr || c->col == nullptr)) return TWELL_ERR_INVALID;
    if (c->backup_cap > 0 && (c->backup_rows == nullptr || c->A_b == nullptr || c->U_b == nullptr))
        return TWELL_ERR_INVALID;
    const void* ps[] = {c->a, c->u, c->col, c->cnt, c->backup_rows, c->n_backup, c->A_b, c->U_b, c->l1, c->dev_status};
    for (const void* p : ps)
        if (p != nullptr && !aligned16(p)) return TWELL_ERR_INVALID;
    if (c->backup_cap > 0 && (static_cast<size_t>(f) * 4) % 16 != 0) return TWELL_ERR_UNSUPPORTED;
    return TWELL_OK;
}

// The fields the routing kernels write (cnt, col, a, backup_rows, n_backup, A_b) and the status
// word; u, U_b and l1 are not touched by routing and may be null.
twell_status check_route_ctx(const twell_hybrid* c, int N, int f, int K)
{
    if (c == nullptr) return TWELL_ERR_INVALID;
    if (c->n_rows != N || c->n_cols != f || c->K != K || c->backup_cap < 0) return TWELL_ERR_INVALID;
    if (c->dtype != TWELL_BF16) return TWELL_ERR_UNSUPPORTED;
    if (N == 0) return TWELL_OK;
    if (c->cnt == nullptr || c->n_backup == nullptr || c->dev_status == nullptr) return TWELL_ERR_INVALID;
    if (K > 0 && (c->a == nullptr || c->col == nullptr)) return TWELL_ERR_INVALID;
    if (c->backup_cap > 0 && (c->backup_rows == nullptr || c->A_b == nullptr)) return TWELL_ERR_INVALID;
    const void* ps[] = {c->a, c->col, c->cnt, c->backup_rows, c->n_backup, c->A_b, c->dev_status};
    for (const void* p : ps)
        if (p != nullptr && !aligned16(p)) return TWELL_ERR_INVALID;
    if (c->backup_cap > 0 && (static_cast<size_t>(f) * 4) % 16 != 0) return TWELL_ERR_UNSUPPORTED;
    return TWELL_OK;
}

inline unsigned grid_for(long long work, int threads, int cap_blocks)
{
    long long g = (work + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > cap_blocks) g = cap_blocks;
    return static_cast<unsigned>(g);
}

// Routing of a gate TwELL (in the workspace) into ctx; gathers x_b when x != nullptr.
twell_status run_route(const twell::HybridWs& L, uint8_t* ws, int N, int f, int K, const bf* x, int d,
                       const twell_hybrid* c, cudaStream_t s)
{
    const float* vals = reinterpret_cast<const float*>(ws + L.tw_vals);
    const uint8_t* idx = ws + L.tw_idx;
    const uint16_t* cnt = reinterpret_cast<const uint16_t*>(ws + L.tw_cnt);
    int* blk = reinterpret_cast<int*>(ws + L.blk);
    double* l1acc = reinterpret_cast<double*>(ws + L.l1acc);
    if (launch_dep(twell::route_rows_kernel, dim3(L.nblk), dim3(32 * twell::kRouteWarps), 0, s,
        vals, idx, cnt, N, f, L.nt, K, static_cast<float*>(c->a), c->col, c->cnt, blk, l1acc, c->dev_status) != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_dep(twell::route_backup_kernel, dim3(L.nblk), dim3(256), 0, s, vals, idx, cnt, c->cnt, blk, L.nblk, N, f, L.nt, c->backup_cap, x,
                                                      d, c->backup_rows, c->n_backup, static_cast<float*>(c->A_b),
                                                      reinterpret_cast<bf*>(ws + L.x_b), c->dev_status) != TWELL_OK) return TWELL_ERR_CUDA;
    return launch_status();
}

}  // namespace

extern "C" size_t twell_workspace_bytes(twell_op op, int32_t N, int32_t d, int32_t f, int32_t tile, int32_t K,
                                        int32_t backup_cap)
{
    if (N < 0 || d <= 0 || f <= 0 || K < 0 || backup_cap < 0) return 0;
    switch (op) {
    case TWELL_OP_GATE_PACK: return 0;
    case TWELL_OP_FFN_FUSED_FWD: return twell_host::fused_ws_bytes(N, d, f);
    case TWELL_OP_FFN_UNION_FWD: return twell_host::union_ws_bytes(N, d, f);
    case TWELL_OP_FFN_TILE_UNION_FWD: return twell_host::tile_union_ws_bytes(N, f);
    case TWELL_OP_FFN_GATE_UNION_FWD: return twell_host::gate_union_ws_bytes(N, d, f);
    case TWELL_OP_FFN_DECODE: return tile > 0 ? twell_host::decode_ws_bytes(N, d, f, tile) : 0;
    case TWELL_OP_HYBRID_ROUTE: return twell::HybridWs(N, d, f, K, backup_cap).route_total;
    case TWELL_OP_HYBRID_FWD: return twell::HybridWs(N, d, f, K, backup_cap).fwd_total;
    case TWELL_OP_HYBRID_BWD: return twell::HybridWs(N, d, f, K, backup_cap).bwd_total;
    }
    return 0;
}

extern "C" twell_status twell_hybrid_route_from_gate(const void* G, int32_t N, int32_t f, int32_t K, twell_dtype dtype,
                                                     const twell_hybrid* ctx, void* ws, size_t ws_bytes, void* stream)
{
    if (dtype != TWELL_BF16) return TWELL_ERR_UNSUPPORTED;
    if (N < 0 || f <= 0 || f > 65535 || K < 0 || K > twell::kMaxK) return TWELL_ERR_INVALID;
    twell_status st = check_hybrid(ctx, N, f, K);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    if (G == nullptr || !aligned16(G)) return TWELL_ERR_INVALID;
    const twell::HybridWs L(N, 8, f, K, ctx->backup_cap);
    if (ws == nullptr || ws_bytes < L.route_total || !aligned16(ws)) return TWELL_ERR_WORKSPACE;
    uint8_t* w = static_cast<uint8_t*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    twell_packed tp{N, f, twell::kHybTile, twell::kHybTile, TWELL_F32, w + L.tw_vals, w + L.tw_idx,
                    reinterpret_cast<uint16_t*>(w + L.tw_cnt)};
    st = pack_gate_widened(G, N, f, &tp, ctx->dev_status, s);
    if (st != TWELL_OK) return st;
    return run_route(L, w, N, f, K, nullptr, 8, ctx, s);
}

extern "C" twell_status twell_hybrid_fwd(const void* x, const void* Wg_s, const void* Wu_s, const void* Wd_s,
                                         int32_t N, int32_t d, int32_t f, int32_t K, float l1_coef, twell_dtype dtype,
                                         const twell_hybrid* ctx, void* y, void* ws, size_t ws_bytes, void* stream)
{
    if (dtype != TWELL_BF16) return TWELL_ERR_UNSUPPORTED;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0 || f % 64 != 0 || f > 65535 || K < 0 || K > twell::kMaxK)
        return TWELL_ERR_INVALID;
    if (d / 8 > 512) return TWELL_ERR_UNSUPPORTED;
    if (Wg_s == nullptr || Wu_s == nullptr || Wd_s == nullptr) return TWELL_ERR_INVALID;
    twell_status st = check_hybrid(ctx, N, f, K);
    if (st != TWELL_OK) return st;
    if (N == 0) return TWELL_OK;
    if (x == nullptr || y == nullptr || ctx->l1 == nullptr) return TWELL_ERR_INVALID;
    if (!aligned16(x) || !aligned16(y) || !aligned16(Wg_s) || !aligned16(Wu_s) || !aligned16(Wd_s))
        return TWELL_ERR_INVALID;
    const int cap = ctx->backup_cap;
    const twell::HybridWs L(N, d, f, K, cap);
    if (ws == nullptr || ws_bytes < L.fwd_total || !aligned16(ws)) return TWELL_ERR_WORKSPACE;
    uint8_t* w = static_cast<uint8_t*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DevInfo di;
    if (dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;

    // 1. gate GEMM + ReLU + TwELL pack (fp32 values) into the workspace
    twell_packed tp{N, f, twell::kHybTile, twell::kHybTile, TWELL_F32, w + L.tw_vals, w + L.tw_idx,
                    reinterpret_cast<uint16_t*>(w + L.tw_cnt)};
    st = twell_gate_pack(x, Wg_s, N, d, f, twell::kHybTile, TWELL_BF16, &tp, nullptr, 0, ctx->dev_status, s);
    if (st != TWELL_OK) return st;
    // 2. routing: sparse block, backup list (ascending rows), A_b and x_b
    st = run_route(L, w, N, f, K, static_cast<const bf*>(x), d, ctx, s);
    if (st != TWELL_OK) return st;
    double* l1acc = reinterpret_cast<double*>(w + L.l1acc);
    // 3. light rows: the tensor-core walk where d_model allows, else one CTA per row
    st = light_fwd_bulk(x, Wu_s, Wd_s, N, d, f, K, static_cast<const float*>(ctx->a), ctx->col, ctx->cnt,
                        static_cast<float*>(ctx->u), y, l1acc, reinterpret_cast<int*>(w + L.tick), ctx->dev_status, s);
    if (st == TWELL_ERR_UNSUPPORTED) {
        const int threads = (d / 8 + 31) / 32 * 32;
        if (launch_dep(twell::hybrid_light_fwd_kernel, dim3(grid_for(N, 1, di.sm_count * 4)), dim3(threads), 0, s,
            static_cast<const bf*>(x), static_cast<const bf*>(Wu_s), static_cast<const bf*>(Wd_s), N, d, f, K,
            static_cast<const float*>(ctx->a), ctx->col, ctx->cnt, static_cast<float*>(ctx->u), static_cast<bf*>(y),
            l1acc, ctx->dev_status) != TWELL_OK) return TWELL_ERR_CUDA;
        st = launch_status();
    }
    if (st != TWELL_OK) return st;
    // 4-6. backup rows: U_b = x_b Wu_s^T, H_b = A_b * U_b, y[rows] = H_b Wd_s
    if (cap > 0) {
        bf* x_b = reinterpret_cast<bf*>(w + L.x_b);
        bf* H_b = reinterpret_cast<bf*>(w + L.h_b);
        twell::GemmArgs g{};
        g.pdl = 1;  // prologue overlaps the previous kernel's tail
        g.M = cap;
        g.N = f;
        g.K = d;
        g.M_dyn = ctx->n_backup;
        g.out = ctx->U_b;
        g.ldo = f;
        g.status = ctx->dev_status;
        st = launch_gemm<256, false, false, twell::Epi::StoreF32>(GemmOperand{x_b, (int64_t)L.capr, d, d},
                                                                  GemmOperand{Wu_s, f, d, d}, nullptr, g, s);
        if (st != TWELL_OK) return st;
        if (launch_dep(twell::backup_h_kernel, dim3(grid_for(static_cast<long long>(cap) * L.f_pad, 256, di.sm_count * 8)), dim3(256), 0, s,
            static_cast<const float*>(ctx->A_b), static_cast<const float*>(ctx->U_b), ctx->n_backup, cap, f, L.f_pad,
            H_b, l1acc) != TWELL_OK) return TWELL_ERR_CUDA;
        if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
        // y[rows] = [h_hi | h_lo] [Wd_s ; Wd_s]: kBackupSplits K ranges into fp32 partials, added
        // up in order into the bf16 rows
        float* y_part = reinterpret_cast<float*>(w + L.y_part);
        twell::GemmArgs g2{};
        g2.pdl = 1;  // prologue overlaps the previous kernel's tail
        g2.M = cap;
        g2.N = d;
        g2.K = 2 * L.f_pad;
        g2.kb_split = L.f_pad / 64;
        g2.k_splits = twell::kBackupSplits;
        g2.split_stride = static_cast<int64_t>(L.capr) * d;
        g2.M_dyn = ctx->n_backup;
        g2.out = y_part;
        g2.ldo = d;
        g2.status = ctx->dev_status;
        const GemmOperand Bd{Wd_s, f, d, d};
        st = launch_gemm<256, false, true, twell::Epi::StoreF32>(
            GemmOperand{H_b, (int64_t)L.capr, 2 * L.f_pad, 2 * L.f_pad}, Bd, &Bd, g2, s);
        if (st != TWELL_OK) return st;
        if (launch_dep(twell::reduce_rows_kernel<bf>, dim3(grid_for(static_cast<long long>(cap) * d / 4, 256, di.sm_count * 8)), dim3(256), 0, s,
            y_part, twell::kBackupSplits, static_cast<long long>(L.capr) * d, ctx->n_backup, cap, d, ctx->backup_rows,
            static_cast<bf*>(y)) != TWELL_OK) return TWELL_ERR_CUDA;
        if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    }
    // 7. L1 term
    if (launch_dep(twell::l1_finalize_kernel, dim3(1), dim3(1), 0, s, l1acc, static_cast<float>(static_cast<double>(l1_coef) /
                                                                         (static_cast<double>(N) * f)),
                                              ctx->l1) != TWELL_OK) return TWELL_ERR_CUDA;
    return launch_status();
}

extern "C" twell_status twell_hybrid_bwd(const void* x, const void* Wg_s, const void* Wu_s, const void* Wd_s,
                                         const twell_hybrid* ctx, const void* dy, int32_t N, int32_t d, int32_t f,
                                         float l1_coef, float* dx, float* dWg_s, float* dWu_s, float* dWd_s, void* ws,
                                         size_t ws_bytes, void* stream)
{
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0 || f % 64 != 0 || f > 65535) return TWELL_ERR_INVALID;
    if (d / 8 > 512) return TWELL_ERR_UNSUPPORTED;
    if (Wg_s == nullptr || Wu_s == nullptr || Wd_s == nullptr || dWg_s == nullptr || dWu_s == nullptr ||
        dWd_s == nullptr)
        return TWELL_ERR_INVALID;
    if (ctx == nullptr) return TWELL_ERR_INVALID;
    const int K = ctx->K;
    if (K < 0 || K > twell::kMaxK) return TWELL_ERR_INVALID;
    twell_status st = check_hybrid(ctx, N, f, K);
    if (st != TWELL_OK) return st;
    if (!aligned16(Wg_s) || !aligned16(Wu_s) || !aligned16(Wd_s) || !aligned16(dWg_s) || !aligned16(dWu_s) ||
        !aligned16(dWd_s))
        return TWELL_ERR_INVALID;
    if (N > 0 && (x == nullptr || dy == nullptr || dx == nullptr || !aligned16(x) || !aligned16(dy) || !aligned16(dx)))
        return TWELL_ERR_INVALID;
    const int cap = ctx->backup_cap;
    const twell::HybridWs L(N, d, f, K, cap);
    if (ws == nullptr || ws_bytes < L.bwd_total || !aligned16(ws)) return TWELL_ERR_WORKSPACE;
    uint8_t* w = static_cast<uint8_t*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DevInfo di;
    if (dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    const float l1_scale = N > 0 ? static_cast<float>(static_cast<double>(l1_coef) / (static_cast<double>(N) * f)) : 0.f;
    const int threads = (d / 8 + 31) / 32 * 32;
    float* ent = reinterpret_cast<float*>(w + L.ent);
    int* ccount = reinterpret_cast<int*>(w + L.ccount);
    int* coff = reinterpret_cast<int*>(w + L.coff);
    int* ccur = reinterpret_cast<int*>(w + L.ccur);
    twell::EntRec* rec = reinterpret_cast<twell::EntRec*>(w + L.rec);

    // 1. light rows: dh, du, dg per entry and dx_r (the tensor-core walk where d_model allows)
    if (N > 0) {
        st = light_bwd_bulk(dy, Wg_s, Wu_s, Wd_s, N, d, f, K, static_cast<const float*>(ctx->a),
                            static_cast<const float*>(ctx->u), ctx->col, ctx->cnt, l1_scale, ent, dx,
                            reinterpret_cast<int*>(w + L.btick), ctx->dev_status, s);
        if (st == TWELL_ERR_UNSUPPORTED) {
            if (launch_dep(twell::hybrid_light_bwd_kernel, dim3(grid_for(N, 1, di.sm_count * 4)), dim3(threads), 0, s,
                static_cast<const bf*>(dy), static_cast<const bf*>(Wg_s), static_cast<const bf*>(Wu_s),
                static_cast<const bf*>(Wd_s), N, d, f, K, static_cast<const float*>(ctx->a),
                static_cast<const float*>(ctx->u), ctx->col, ctx->cnt, l1_scale, ent, dx, ctx->dev_status) != TWELL_OK) return TWELL_ERR_CUDA;
            st = launch_status();
        }
        if (st != TWELL_OK) return st;
    }
    // 2. column records of the kept entries (light rows from the sparse block, backup rows from
    //    their dense a), per hidden unit, for the weight gradients
    const long long ne = static_cast<long long>(N) * K;
    const bool backup = cap > 0 && N > 0;
    if (launch_dep(twell::fill_i32_kernel, dim3(grid_for(f, 256, 256)), dim3(256), 0, s, ccount, f, 0) != TWELL_OK) return TWELL_ERR_CUDA;
    if (ne > 0)
        if (launch_dep(twell::col_hist_kernel, dim3(grid_for(ne, 256, di.sm_count * 8)), dim3(256), 0, s, ctx->col, ctx->cnt, N, K, f, ccount) != TWELL_OK) return TWELL_ERR_CUDA;
    if (backup)
        if (launch_dep(twell::col_hist_backup_kernel, dim3(grid_for(static_cast<long long>(cap) * f, 256, di.sm_count * 8)), dim3(256), 0, s,
            static_cast<const float*>(ctx->A_b), ctx->n_backup, cap, f, ccount) != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_dep(twell::col_scan_kernel, dim3(1), dim3(1024), 0, s, ccount, f, coff, ccur) != TWELL_OK) return TWELL_ERR_CUDA;
    if (ne > 0)
        if (launch_dep(twell::col_scatter_kernel, dim3(grid_for(ne, 256, di.sm_count * 8)), dim3(256), 0, s, ctx->col, ctx->cnt, N, K, f, ent,
                                                                                     ccur, rec) != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;

    // 3. backup rows: dH_b = dy_b Wd_s^T (tcgen05), then du, dg (and their column records)
    bf* dy_b = reinterpret_cast<bf*>(w + L.dy_b);
    float* dH = reinterpret_cast<float*>(w + L.dh_b);
    bf* DUG = reinterpret_cast<bf*>(w + L.dug);
    if (backup) {
        const unsigned gg = grid_for(static_cast<long long>(L.capr) * d / 8, 256, di.sm_count * 8);
        if (launch_dep(twell::gather_rows_kernel, dim3(gg), dim3(256), 0, s, static_cast<const bf*>(dy), ctx->backup_rows, ctx->n_backup, cap,
                                                     d, dy_b) != TWELL_OK) return TWELL_ERR_CUDA;
        if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
        twell::GemmArgs g{};
        g.pdl = 1;  // prologue overlaps the previous kernel's tail
        g.M = cap;
        g.N = f;
        g.K = d;
        g.M_dyn = ctx->n_backup;
        g.out = dH;
        g.ldo = L.f_pad;
        g.status = ctx->dev_status;
        st = launch_gemm<256, false, false, twell::Epi::StoreF32>(GemmOperand{dy_b, (int64_t)L.capr, d, d},
                                                                  GemmOperand{Wd_s, f, d, d}, nullptr, g, s);
        if (st != TWELL_OK) return st;
        if (launch_dep(twell::backup_grad_kernel, dim3(grid_for(static_cast<long long>(L.capr) * L.f_pad, 256, di.sm_count * 8)), dim3(256), 0, s, static_cast<const float*>(ctx->A_b), static_cast<const float*>(ctx->U_b), dH,
                                         ctx->n_backup, cap, f, L.f_pad, l1_scale, ctx->backup_rows, ccur, rec, DUG) != TWELL_OK) return TWELL_ERR_CUDA;
        if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    }

    // 4. weight gradients of every kept entry, per hidden unit, in row order (overwrites dW)
    if (launch_dep(twell::col_sort_kernel, dim3(grid_for(f, 128, di.sm_count * 4)), dim3(128), 0, s, coff, f, rec) != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_dep(twell::col_dw_kernel<0>, dim3(f), dim3(threads), 0, s,
        coff, rec, f, d, static_cast<const bf*>(x), dWg_s, dWu_s) != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_dep(twell::col_dw_kernel<1>, dim3(f), dim3(threads), 0, s,
        coff, rec, f, d, static_cast<const bf*>(dy), dWd_s, nullptr) != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    if (!backup) return TWELL_OK;

    // 5. dx[rows] = [du_hi | dg_hi | du_lo | dg_lo] [Wu_s ; Wg_s ; Wu_s ; Wg_s] (fp32 output), in
    //    kBackupSplits K ranges added up in order
    float* dx_part = reinterpret_cast<float*>(w + L.dx_part);
    twell::GemmArgs g{};
    g.pdl = 1;  // prologue overlaps the previous kernel's tail
    g.M = cap;
    g.N = d;
    g.K = 4 * L.f_pad;
    g.M_dyn = ctx->n_backup;
    g.kb_split = L.f_pad / 64;
    g.k_splits = twell::kBackupSplits;
    g.split_stride = static_cast<int64_t>(L.capr) * d;
    g.out = dx_part;
    g.ldo = d;
    g.status = ctx->dev_status;
    const GemmOperand B2{Wg_s, f, d, d};
    st = launch_gemm<256, false, true, twell::Epi::StoreF32>(GemmOperand{DUG, (int64_t)L.capr, 4 * L.f_pad, 4 * L.f_pad},
                                                             GemmOperand{Wu_s, f, d, d}, &B2, g, s);
    if (st != TWELL_OK) return st;
    if (launch_dep(twell::reduce_rows_kernel<float>, dim3(grid_for(static_cast<long long>(cap) * d / 4, 256, di.sm_count * 8)), dim3(256), 0, s,
        dx_part, twell::kBackupSplits, static_cast<long long>(L.capr) * d, ctx->n_backup, cap, d, ctx->backup_rows, dx) != TWELL_OK) return TWELL_ERR_CUDA;
    return launch_status();
}

// Test export: C = A * B in fp32 from the tcgen05 GEMM with any operand major-ness.
extern "C" twell_status twell_gemm_test(const void* A, const void* B, int32_t M, int32_t N, int32_t K, int32_t a_mn,
                                        int32_t b_mn, float* C, int32_t* dev_status, void* stream)
{
    if (A == nullptr || B == nullptr || C == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if (M <= 0 || N <= 0 || K <= 0 || N % 8 != 0 || (a_mn ? M : K) % 8 != 0 || (b_mn ? N : K) % 8 != 0)
        return TWELL_ERR_INVALID;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return TWELL_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    twell::GemmArgs g{};
    g.M = M;
    g.N = N;
    g.K = K;
    g.out = C;
    g.ldo = N;
    g.status = dev_status;
    const GemmOperand Ao = a_mn ? GemmOperand{A, K, M, M} : GemmOperand{A, M, K, K};
    const GemmOperand Bo = b_mn ? GemmOperand{B, K, N, N} : GemmOperand{B, N, K, K};
    if (!a_mn && !b_mn) return launch_gemm<256, false, false, twell::Epi::StoreF32>(Ao, Bo, nullptr, g, s);
    if (a_mn && !b_mn) return launch_gemm<256, true, false, twell::Epi::StoreF32>(Ao, Bo, nullptr, g, s);
    if (!a_mn && b_mn) return launch_gemm<256, false, true, twell::Epi::StoreF32>(Ao, Bo, nullptr, g, s);
    return launch_gemm<256, true, true, twell::Epi::StoreF32>(Ao, Bo, nullptr, g, s);
}

// ------------------------------------------------------------------------------------------
// Routing without any allocation or workspace.
//
// Some callers cannot hand the library a workspace or let anything allocate device memory: code
// living inside a framework whose caching allocator owns all device memory (a second allocator
// would fight it for the same HBM), plug-in hosts that pass only inputs and outputs across their
// interface, and latency-critical loops where a cudaMalloc / cudaFree would synchronise the
// device. For them the routing of an already packed TwELL matrix keeps its only scratch -- the
// number of overflow rows of each 128-row block -- in the fixed array below. The array lives in
// every GPU that loads the library until the process exits, and holds the previous call's counts;
// nothing in it has to start at zero, because the first kernel of every call rewrites each entry
// the second kernel reads. Calls that overlap on the GPU share the array and race.

namespace {

constexpr int kNoAllocBlocks = 32768;  // 32-row blocks: at most 1,048,576 token rows per call
static __device__ __align__(256) int32_t g_noalloc_blk_counts[kNoAllocBlocks];

std::mutex g_noalloc_mu;
int32_t* g_noalloc_ptr[64] = {};

// Device address of the array on the current device, looked up once per device.
twell_status noalloc_scratch(int32_t** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TWELL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_blk_counts) != cudaSuccess || p == nullptr) return TWELL_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return TWELL_OK;
}

}  // namespace

extern "C" twell_status twell_hybrid_route_noalloc(const twell_packed* a, int32_t K, const twell_hybrid* ctx,
                                                   void* stream)
{
    if (a == nullptr || ctx == nullptr) return TWELL_ERR_INVALID;
    const int N = a->n_rows, f = a->n_cols;
    if (N < 0 || f <= 0 || f > 65535 || K < 0 || K > twell::kMaxK) return TWELL_ERR_INVALID;
    if (a->dtype != TWELL_F32 || a->tile != twell::kHybTile) return TWELL_ERR_UNSUPPORTED;
    twell_status st = check_packed(a, N, f, twell::kHybTile, TWELL_F32);
    if (st != TWELL_OK) return st;
    st = check_route_ctx(ctx, N, f, K);
    if (st != TWELL_OK) return st;
    const int nblk = (N + twell::kRouteRows - 1) / twell::kRouteRows;
    if (nblk > kNoAllocBlocks) return TWELL_ERR_UNSUPPORTED;  // more rows than the fixed scratch covers
    if (N == 0) return TWELL_OK;
    int32_t* blk = nullptr;
    st = noalloc_scratch(&blk);
    if (st != TWELL_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int nt = (f + twell::kHybTile - 1) / twell::kHybTile;
    if (launch_dep(twell::route_rows_kernel, dim3(nblk), dim3(32 * twell::kRouteWarps), 0, s,
        static_cast<const float*>(a->vals), a->idx, a->cnt, N, f, nt, K, static_cast<float*>(ctx->a), ctx->col, ctx->cnt,
        blk, nullptr, ctx->dev_status) != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    if (launch_dep(twell::route_backup_kernel, dim3(nblk), dim3(256), 0, s, static_cast<const float*>(a->vals), a->idx, a->cnt, ctx->cnt, blk,
                                                    nblk, N, f, nt, ctx->backup_cap, nullptr, 8, ctx->backup_rows,
                                                    ctx->n_backup, static_cast<float*>(ctx->A_b), nullptr,
                                                    ctx->dev_status) != TWELL_OK) return TWELL_ERR_CUDA;
    return launch_status();
}
