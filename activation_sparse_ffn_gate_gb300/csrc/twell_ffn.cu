// twell_ffn.cu -- fused up+down projection over a TwELL matrix of gate activations.
//
// For every token row r the kernel walks only the packed nonzeros (column j, value a) of that
// row, gathers row j of Wu_s and row j of Wd_s, forms u = x_r . Wu_s[j], h = a * u and
// accumulates y_r += h * Wd_s[j] in fp32 registers; the hidden activation never leaves the SM
// ([AIM] ¶3; [TG] "Инференс"; [PUL] ¶3; [TC] §2).
//
// GB300 layout: one persistent CTA per SM, rows assigned round-robin. The CTA is split into
//   - a producer warp that reads the TwELL counts/indices of its rows, and streams the needed
//     weight rows (Wu_s[j] and Wd_s[j], d*2 bytes each) and each row's x into shared-memory
//     rings with cp.async.bulk copies completing on mbarriers (weights with an L2 evict-last
//     hint so they stay resident, x with evict-first). It runs up to S nonzeros ahead, across
//     row boundaries, so ~S*4*d bytes of gathers are always in flight;
//   - consumer warps (one thread per 16-byte chunk of d_model) that take the staged nonzeros in
//     batches of kBatch: each thread forms its chunk's partial dots with x_r, the dots are reduced
//     with warp shuffles and one named barrier (which also agrees on abort), and each thread
//     applies the kBatch rank-1 updates h * Wd_s[j] to its fp32 slice of y_r, then frees the slots.
// Every wait is bounded; on a timeout the CTA records TWELL_ERR_TIMEOUT, all roles leave their
// loops together, and the producer waits (bounded) for its copies in flight before exit.
#include "twell_common.cuh"

namespace twell {

constexpr int kBatch = 8;
constexpr int kListCap = 256;
constexpr int kMaxTiles = 1024;
constexpr int kRowSlots = 4;
constexpr int kMaxSlots = 32;
constexpr int kMaxConsumers = 512;

template <typename E, typename VT>
struct FusedArgs {
    const E* x;
    const E* Wu;
    const E* Wd;
    const VT* vals;
    const uint8_t* idx;
    const uint16_t* cnt;
    E* y;
    int N, d, f, T, nt;
    int S;          // weight-row slots in the ring
    int consumers;  // consumer threads (multiple of 32)
    int32_t* status;
    uint64_t wait_limit_ns;
};

struct FusedLayout {
    size_t wu, wd, x, a, nnz, pref, lj, la, red, bars, abort_flag, total;
    __host__ __device__ FusedLayout(int S, int row_bytes)
    {
        size_t o = 0;
        wu = o;
        o += static_cast<size_t>(S) * row_bytes;
        wd = o;
        o += static_cast<size_t>(S) * row_bytes;
        x = o;
        o += static_cast<size_t>(kRowSlots) * row_bytes;
        a = o;
        o += kMaxSlots * 4;
        nnz = o;
        o += kRowSlots * 4;
        pref = o;
        o += (kMaxTiles + 1) * 4;
        lj = o;
        o += kListCap * 4;
        la = o;
        o += kListCap * 4;
        red = o;
        o += 2 * (kMaxConsumers / 32) * kBatch * 4;
        o = (o + 7) & ~size_t(7);
        bars = o;
        o += (2 * kMaxSlots + 2 * kRowSlots) * 8;
        abort_flag = o;
        o += 16;
        total = o;
    }
};

template <typename E, typename VT, int CPT>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1) ffn_fused_kernel(const FusedArgs<E, VT> a)
{
    constexpr int V = Elem<E>::kPer16B;
    extern __shared__ __align__(128) uint8_t smem[];
    const int row_bytes = a.d * static_cast<int>(sizeof(E));
    const FusedLayout L(a.S, row_bytes);
    E* s_wu = reinterpret_cast<E*>(smem + L.wu);
    E* s_wd = reinterpret_cast<E*>(smem + L.wd);
    E* s_x = reinterpret_cast<E*>(smem + L.x);
    float* s_a = reinterpret_cast<float*>(smem + L.a);
    int* s_nnz = reinterpret_cast<int*>(smem + L.nnz);
    int* s_pref = reinterpret_cast<int*>(smem + L.pref);
    int* s_lj = reinterpret_cast<int*>(smem + L.lj);
    float* s_la = reinterpret_cast<float*>(smem + L.la);
    float* s_red = reinterpret_cast<float*>(smem + L.red);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + kMaxSlots;
    uint64_t* rfull = empty + kMaxSlots;
    uint64_t* rempty = rfull + kRowSlots;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int C = a.consumers;
    const int cwarps = C >> 5;
    const int S = a.S;
    const int nchunks = a.d / V;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], cwarps);
        }
        for (int s = 0; s < kRowSlots; ++s) {
            mbar_init(&rfull[s], 1);
            mbar_init(&rempty[s], cwarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (tid >= C) {
        // ---------------------------------------------------------------- producer warp
        const uint64_t pol_w = policy_evict_last();
        const uint64_t pol_x = policy_evict_first();
        int slot = 0, rs = 0;
        uint32_t ph = 0, rph = 0;
        uint32_t issued = 0, issued_ph = 0, xissued = 0, xissued_ph = 0;
        bool ok = true;
        for (int r = blockIdx.x; ok && r < a.N; r += gridDim.x) {
            // exclusive prefix of the row's per-tile counts
            int run = 0;
            for (int t0 = 0; t0 < a.nt; t0 += 32) {
                const int t = t0 + lane;
                int c = t < a.nt ? static_cast<int>(a.cnt[static_cast<size_t>(r) * a.nt + t]) : 0;
                if (c > a.T) {
                    report(a.status, TWELL_ERR_DEVICE_CHECK);
                    c = 0;
                }
                int inc = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += v;
                }
                if (t < a.nt) s_pref[t] = run + inc - c;
                run += __shfl_sync(0xffffffffu, inc, 31);
            }
            if (lane == 0) s_pref[a.nt] = run;
            __syncwarp();
            const int nnz = run;
            // row record: nonzero count and the staged x row
            if (lane == 0) {
                ok = wait_bounded(&rempty[rs], rph ^ 1u, abort_flag, a.status, a.wait_limit_ns);
                if (ok) {
                    s_nnz[rs] = nnz;
                    if (nnz > 0) {
                        mbar_arrive_expect_tx(&rfull[rs], row_bytes);
                        bulk_load(s_x + static_cast<size_t>(rs) * a.d, a.x + static_cast<size_t>(r) * a.d, row_bytes,
                                  &rfull[rs], pol_x);
                        xissued |= 1u << rs;
                        xissued_ph = (xissued_ph & ~(1u << rs)) | (rph << rs);
                    } else {
                        mbar_arrive(&rfull[rs]);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            if (++rs == kRowSlots) {
                rs = 0;
                rph ^= 1u;
            }
            // the row's nonzeros, in TwELL order, in windows of kListCap
            for (int base = 0; ok && base < nnz; base += kListCap) {
                const int n = min(kListCap, nnz - base);
                for (int t = lane; t < a.nt; t += 32) {
                    const int s = s_pref[t], e = s_pref[t + 1];
                    const int lo = max(s, base), hi = min(e, base + n);
                    const size_t sb = (static_cast<size_t>(r) * a.nt + t) * a.T;
                    for (int p = lo; p < hi; ++p) {
                        int j = t * a.T + a.idx[sb + (p - s)];
                        float v = Elem<VT>::to_f(a.vals[sb + (p - s)]);
                        if (j >= a.f) {  // corrupt index: record it and contribute nothing
                            report(a.status, TWELL_ERR_DEVICE_CHECK);
                            j = 0;
                            v = 0.0f;
                        }
                        s_lj[p - base] = j;
                        s_la[p - base] = v;
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    for (int p = 0; p < n; ++p) {
                        if (!wait_bounded(&empty[slot], ph ^ 1u, abort_flag, a.status, a.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        const size_t j = static_cast<size_t>(s_lj[p]);
                        s_a[slot] = s_la[p];
                        mbar_arrive_expect_tx(&full[slot], 2 * row_bytes);
                        bulk_load(s_wu + static_cast<size_t>(slot) * a.d, a.Wu + j * a.d, row_bytes, &full[slot], pol_w);
                        bulk_load(s_wd + static_cast<size_t>(slot) * a.d, a.Wd + j * a.d, row_bytes, &full[slot], pol_w);
                        issued |= 1u << slot;
                        issued_ph = (issued_ph & ~(1u << slot)) | (ph << slot);
                        if (++slot == S) {
                            slot = 0;
                            ph ^= 1u;
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                __syncwarp();
            }
        }
        // no bulk copy may still be writing shared memory when the CTA exits
        if (lane == 0) {
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s)) wait_bounded(&full[s], (issued_ph >> s) & 1u, nullptr, a.status, a.wait_limit_ns);
            for (int s = 0; s < kRowSlots; ++s)
                if (xissued & (1u << s))
                    wait_bounded(&rfull[s], (xissued_ph >> s) & 1u, nullptr, a.status, a.wait_limit_ns);
        }
    } else {
        // ---------------------------------------------------------------- consumer warps
        const int warp = tid >> 5;
        int slot = 0, rs = 0, buf = 0;
        uint32_t ph = 0, rph = 0;
        for (int r = blockIdx.x; r < a.N; r += gridDim.x) {
            const bool rok = wait_bounded(&rfull[rs], rph, abort_flag, a.status, a.wait_limit_ns);
            if (bar_or(1, C, !rok)) break;
            const int nnz = s_nnz[rs];
            float acc[CPT][V];
            uint4 xr[CPT];
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int q = tid + i * C;
                xr[i] = (nnz > 0 && q < nchunks)
                            ? *reinterpret_cast<const uint4*>(s_x + static_cast<size_t>(rs) * a.d + q * V)
                            : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int e = 0; e < V; ++e) acc[i][e] = 0.0f;
            }
            bool failed = false;
            for (int b = 0; b < nnz; b += kBatch) {
                const int nb = min(kBatch, nnz - b);
                bool okb = true;
                float pd[kBatch];
                {
                    int s = slot;
                    uint32_t p = ph;
#pragma unroll
                    for (int k = 0; k < kBatch; ++k) {
                        float acc_d = 0.0f;
                        if (k < nb) {
                            okb = okb && wait_bounded(&full[s], p, abort_flag, a.status, a.wait_limit_ns);
#pragma unroll
                            for (int i = 0; i < CPT; ++i) {
                                const int q = tid + i * C;
                                if (q < nchunks) {
                                    float xv[V], wv[V];
                                    unpack16(xr[i], xv, static_cast<E*>(nullptr));
                                    unpack16(*reinterpret_cast<const uint4*>(s_wu + static_cast<size_t>(s) * a.d + q * V),
                                             wv, static_cast<E*>(nullptr));
#pragma unroll
                                    for (int e = 0; e < V; ++e) acc_d = fmaf(xv[e], wv[e], acc_d);
                                }
                            }
                            if (++s == S) {
                                s = 0;
                                p ^= 1u;
                            }
                        }
                        pd[k] = acc_d;
                    }
                }
#pragma unroll
                for (int k = 0; k < kBatch; ++k)
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) pd[k] += __shfl_xor_sync(0xffffffffu, pd[k], o);
                if (lane == 0) {
#pragma unroll
                    for (int k = 0; k < kBatch; ++k) s_red[(buf * (kMaxConsumers / 32) + warp) * kBatch + k] = pd[k];
                }
                if (bar_or(1, C, !okb)) {
                    failed = true;
                    break;
                }
                {
                    int s = slot;
#pragma unroll
                    for (int k = 0; k < kBatch; ++k) {
                        if (k < nb) {
                            float u = 0.0f;
                            for (int w = 0; w < cwarps; ++w) u += s_red[(buf * (kMaxConsumers / 32) + w) * kBatch + k];
                            const float h = s_a[s] * u;
#pragma unroll
                            for (int i = 0; i < CPT; ++i) {
                                const int q = tid + i * C;
                                if (q < nchunks) {
                                    float wv[V];
                                    unpack16(*reinterpret_cast<const uint4*>(s_wd + static_cast<size_t>(s) * a.d + q * V),
                                             wv, static_cast<E*>(nullptr));
#pragma unroll
                                    for (int e = 0; e < V; ++e) acc[i][e] = fmaf(h, wv[e], acc[i][e]);
                                }
                            }
                            if (++s == S) s = 0;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    int s = slot;
                    for (int k = 0; k < nb; ++k) {
                        mbar_arrive(&empty[s]);
                        if (++s == S) s = 0;
                    }
                }
                slot += nb;
                if (slot >= S) {
                    slot -= S;
                    ph ^= 1u;
                }
                buf ^= 1;
            }
            if (failed) break;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int q = tid + i * C;
                if (q < nchunks) st_stream16(a.y + static_cast<size_t>(r) * a.d + q * V, pack16(acc[i], static_cast<E*>(nullptr)));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[rs]);
            if (++rs == kRowSlots) {
                rs = 0;
                rph ^= 1u;
            }
        }
    }
    __syncthreads();
}

template <typename E, typename VT, int CPT>
static twell_status launch_fused(FusedArgs<E, VT> a, cudaStream_t s)
{
    twell_host::DevInfo di;
    if (twell_host::dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    constexpr int V = Elem<E>::kPer16B;
    const int nchunks = a.d / V;
    a.consumers = ((nchunks + CPT - 1) / CPT + 31) / 32 * 32;
    const int row_bytes = a.d * static_cast<int>(sizeof(E));
    const size_t fixed = FusedLayout(0, row_bytes).total;
    const size_t budget = di.max_smem_optin;
    if (budget <= fixed) return TWELL_ERR_UNSUPPORTED;
    int S = static_cast<int>((budget - fixed) / (2 * static_cast<size_t>(row_bytes)));
    if (S > kMaxSlots) S = kMaxSlots;
    if (S < kBatch) return TWELL_ERR_UNSUPPORTED;
    a.S = S;
    a.wait_limit_ns = twell_host::wait_limit_ns();
    const size_t smem = FusedLayout(S, row_bytes).total;
    auto kern = ffn_fused_kernel<E, VT, CPT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return TWELL_ERR_CUDA;
    const int grid = a.N < di.sm_count ? a.N : di.sm_count;
    kern<<<grid, a.consumers + 32, smem, s>>>(a);
    return twell_host::launch_status();
}

template <typename E, typename VT>
static twell_status run_fused(const FusedArgs<E, VT>& a, cudaStream_t s)
{
    constexpr int V = Elem<E>::kPer16B;
    const int nchunks = a.d / V;
    if (nchunks <= kMaxConsumers) return launch_fused<E, VT, 1>(a, s);
    if (nchunks <= 2 * kMaxConsumers) return launch_fused<E, VT, 2>(a, s);
    return TWELL_ERR_UNSUPPORTED;
}

}  // namespace twell

using namespace twell_host;

extern "C" twell_status twell_ffn_fused_fwd(const void* x, const void* Wu_s, const void* Wd_s, const twell_packed* a,
                                            int32_t N, int32_t d, int32_t f, twell_dtype dtype, void* y, void* ws,
                                            size_t ws_bytes, int32_t* dev_status, void* stream)
{
    (void)ws;
    (void)ws_bytes;
    if (Wu_s == nullptr || Wd_s == nullptr || a == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if ((x == nullptr || y == nullptr) && N != 0) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0) return TWELL_ERR_INVALID;
    if (!dtype_ok(dtype) || !dtype_ok(a->dtype)) return TWELL_ERR_UNSUPPORTED;
    if (dtype == TWELL_F32 && a->dtype != TWELL_F32) return TWELL_ERR_INVALID;
    twell_status st = check_packed(a, N, f, a->tile, a->dtype);
    if (st != TWELL_OK) return st;
    const int nt = (f + a->tile - 1) / a->tile;
    if (nt > twell::kMaxTiles) return TWELL_ERR_UNSUPPORTED;
    if (N == 0) return TWELL_OK;
    if (!aligned16(x) || !aligned16(Wu_s) || !aligned16(Wd_s) || !aligned16(y)) return TWELL_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    using bf = __nv_bfloat16;
    if (dtype == TWELL_BF16) {
        const bf* xb = static_cast<const bf*>(x);
        const bf* wu = static_cast<const bf*>(Wu_s);
        const bf* wd = static_cast<const bf*>(Wd_s);
        bf* yb = static_cast<bf*>(y);
        if (a->dtype == TWELL_F32) {
            twell::FusedArgs<bf, float> p{xb, wu, wd, static_cast<const float*>(a->vals), a->idx, a->cnt, yb,
                                          N, d, f, a->tile, nt, 0, 0, dev_status, 0};
            return twell::run_fused(p, s);
        }
        twell::FusedArgs<bf, bf> p{xb, wu, wd, static_cast<const bf*>(a->vals), a->idx, a->cnt, yb,
                                   N, d, f, a->tile, nt, 0, 0, dev_status, 0};
        return twell::run_fused(p, s);
    }
    twell::FusedArgs<float, float> p{static_cast<const float*>(x), static_cast<const float*>(Wu_s),
                                     static_cast<const float*>(Wd_s), static_cast<const float*>(a->vals), a->idx,
                                     a->cnt, static_cast<float*>(y), N, d, f, a->tile, nt, 0, 0, dev_status, 0};
    return twell::run_fused(p, s);
}
