// twell_ffn.cu -- fused up+down projection over a TwELL matrix of gate activations.
//
// For every token row r the kernel walks only the packed nonzeros (column j, value a) of that
// row, gathers row j of Wu_s and row j of Wd_s, forms u = x_r . Wu_s[j], h = a * u and
// accumulates y_r += h * Wd_s[j] in fp32 registers; the hidden activation never leaves the SM
// ([AIM] ¶3; [TG] "Инференс"; [PUL] ¶3; [TC] §2).
//
// GB300 layout: one persistent CTA per SM, rows assigned round-robin. The CTA is split into
//   - a metadata warp that reads the TwELL counts, indices and values of its rows and writes
//     them as an item stream (row record, then the row's nonzeros) into a shared-memory ring,
//     running ahead of use;
//   - an issuer warp that walks the items and streams the needed weight rows (Wu_s[j] and
//     Wd_s[j], d*2 bytes each) and each row's x into shared-memory rings with cp.async.bulk
//     copies completing on mbarriers (weights with an L2 evict-last hint so they stay resident,
//     x with evict-first). It runs up to S nonzeros ahead, across row boundaries, so about
//     S*4*d bytes of gathers are in flight;
//   - consumer warps (one thread per 16-byte chunk of d_model) that take the staged nonzeros in
//     batches of one nonzero per warp: each warp forms the whole dot x_r . Wu_s[j] of its nonzero
//     (warp shuffles only), one named barrier publishes the batch's h = a*u (and agrees on
//     abort), and every thread applies the batch's rank-1 updates h * Wd_s[j] to its fp32 slice
//     of y_r, then frees the slots.
// Every wait is bounded; on a timeout the CTA records TWELL_ERR_TIMEOUT, all roles leave their
// loops together, and the producer waits (bounded) for its copies in flight before exit.
#include "twell_common.cuh"

namespace twell {

constexpr int kItemCap = 256;   // items per buffer of the metadata -> issuer ring
constexpr int kItemBufs = 4;
constexpr int kItemEager = 64;  // a buffer holding this many items is handed over at the next row end
constexpr int kCntRegs = 4;     // rows with nt <= 128 tiles get their counts prefetched in registers
constexpr int kEndItem = -2147483647 - 1;
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

// Shared-memory layout of the fused kernel. Every region starts on a 16-byte boundary (bulk-copy
// destinations need 16 bytes, the item ring holds 8-byte int2, mbarriers need 8).
struct FusedLayout {
    size_t wu, wd, x, a, nnz, pref, items, nitems, red, bars, abort_flag, total;
    __host__ __device__ static size_t up16(size_t v) { return (v + 15) & ~size_t(15); }
    __host__ __device__ FusedLayout(int S, int row_bytes)
    {
        size_t o = 0;
        wu = o;
        o = up16(o + static_cast<size_t>(S) * row_bytes);
        wd = o;
        o = up16(o + static_cast<size_t>(S) * row_bytes);
        x = o;
        o = up16(o + static_cast<size_t>(kRowSlots) * row_bytes);
        a = o;
        o = up16(o + kMaxSlots * 4);
        nnz = o;
        o = up16(o + kRowSlots * 4);
        pref = o;
        o = up16(o + (kMaxTiles + 1) * 4);
        items = o;
        o = up16(o + kItemBufs * kItemCap * 8);
        nitems = o;
        o = up16(o + kItemBufs * 4);
        red = o;
        o = up16(o + 2 * (kMaxConsumers / 32) * 4);
        bars = o;
        o = up16(o + (2 * kMaxSlots + 2 * kRowSlots + 2 * kItemBufs) * 8);
        abort_flag = o;
        o = up16(o + 16);
        total = o;
    }
    __host__ bool aligned() const
    {
        const size_t all[] = {wu, wd, x, a, nnz, pref, items, nitems, red, bars, abort_flag, total};
        for (size_t v : all)
            if (v % 16 != 0) return false;
        return true;
    }
};

// Threads per CTA: consumer warps (<= XC of them when x is held in registers) + 2 producer warps.
template <int XC>
struct FusedThreads {
    static constexpr int kMax = (XC > 0 ? 32 * XC : kMaxConsumers) + 64;
};

template <typename E, typename VT, int XC>
__global__ void __launch_bounds__(FusedThreads<XC>::kMax, 1) ffn_fused_kernel(const FusedArgs<E, VT> a)
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
    int2* s_items = reinterpret_cast<int2*>(smem + L.items);
    int* s_nitems = reinterpret_cast<int*>(smem + L.nitems);
    float* s_red = reinterpret_cast<float*>(smem + L.red);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + kMaxSlots;
    uint64_t* rfull = empty + kMaxSlots;
    uint64_t* rempty = rfull + kRowSlots;
    uint64_t* lfull = rempty + kRowSlots;
    uint64_t* lempty = lfull + kItemBufs;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_flag);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int C = a.consumers;
    const int cwarps = C >> 5;
    const int S = a.S;
    const int batch = min(cwarps, S);  // nonzeros per consumer batch (one per warp)
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
        for (int s = 0; s < kItemBufs; ++s) {
            mbar_init(&lfull[s], 1);
            mbar_init(&lempty[s], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (tid >= C + 32) {
        // ---------------------------------------------------------------- metadata warp
        // Turns the TwELL of this CTA's rows into a stream of items for the issuer: a row record
        // {~r, nnz} followed by the row's nonzeros {j, a} in TwELL order, written into a ring of
        // kItemBufs buffers. The counts of the next row are loaded while the current row's
        // indices and values are gathered, so one L2 round trip is paid per row, ahead of use.
        int buf = 0, fill = 0;
        uint32_t bph = 0;
        bool ok = true;
        auto publish = [&]() {  // hand the current buffer to the issuer and open the next one
            __syncwarp();
            if (lane == 0) {
                s_nitems[buf] = fill;
                mbar_arrive(&lfull[buf]);
            }
            if (++buf == kItemBufs) {
                buf = 0;
                bph ^= 1u;
            }
            fill = 0;
            int w = 1;
            if (lane == 0) w = wait_bounded(&lempty[buf], bph ^ 1u, abort_flag, a.status, a.wait_limit_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        };
        {
            int w = 1;
            if (lane == 0) w = wait_bounded(&lempty[0], 1u, abort_flag, a.status, a.wait_limit_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        }
        const bool pre = a.nt <= 32 * kCntRegs;
        int creg[kCntRegs];
        auto load_counts = [&](int row, int (&c)[kCntRegs]) {
#pragma unroll
            for (int m = 0; m < kCntRegs; ++m) {
                const int t = lane + 32 * m;
                c[m] = (row < a.N && t < a.nt) ? static_cast<int>(a.cnt[static_cast<size_t>(row) * a.nt + t]) : 0;
            }
        };
        if (pre) load_counts(blockIdx.x, creg);
        for (int r = blockIdx.x; ok && r < a.N; r += gridDim.x) {
            // per-tile exclusive offsets of row r in shared memory
            int run = 0;
            if (pre) {
                int c[kCntRegs];
#pragma unroll
                for (int m = 0; m < kCntRegs; ++m) c[m] = creg[m];
                load_counts(r + gridDim.x, creg);  // next row's counts, in flight during this row
#pragma unroll
                for (int m = 0; m < kCntRegs; ++m) {
                    const int t = lane + 32 * m;
                    int v = c[m];
                    if (v > a.T) {
                        report(a.status, TWELL_ERR_DEVICE_CHECK);
                        v = 0;
                    }
                    int inc = v;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int u = __shfl_up_sync(0xffffffffu, inc, o);
                        if (lane >= o) inc += u;
                    }
                    if (t < a.nt) s_pref[t] = run + inc - v;
                    run += __shfl_sync(0xffffffffu, inc, 31);
                }
            } else {
                for (int t0 = 0; t0 < a.nt; t0 += 32) {
                    const int t = t0 + lane;
                    int v = t < a.nt ? static_cast<int>(a.cnt[static_cast<size_t>(r) * a.nt + t]) : 0;
                    if (v > a.T) {
                        report(a.status, TWELL_ERR_DEVICE_CHECK);
                        v = 0;
                    }
                    int inc = v;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int u = __shfl_up_sync(0xffffffffu, inc, o);
                        if (lane >= o) inc += u;
                    }
                    if (t < a.nt) s_pref[t] = run + inc - v;
                    run += __shfl_sync(0xffffffffu, inc, 31);
                }
            }
            if (lane == 0) s_pref[a.nt] = run;
            __syncwarp();
            const int nnz = run;
            if (fill == kItemCap) publish();
            if (!ok) break;
            if (lane == 0) s_items[buf * kItemCap + fill] = make_int2(~r, nnz);
            ++fill;
            for (int pos = 0; ok && pos < nnz;) {
                if (fill == kItemCap) {
                    publish();
                    if (!ok) break;
                }
                const int take = min(kItemCap - fill, nnz - pos);
                // one entry per lane: its tile is the last t with s_pref[t] <= position (binary
                // search), so all the row's index/value loads are in flight together
                for (int i = lane; i < take; i += 32) {
                    const int gp = pos + i;
                    int lo = 0, hi = a.nt;  // invariant: s_pref[lo] <= gp < s_pref[hi]
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (s_pref[mid] <= gp) lo = mid;
                        else hi = mid;
                    }
                    const size_t e = (static_cast<size_t>(r) * a.nt + lo) * a.T + (gp - s_pref[lo]);
                    int j = lo * a.T + a.idx[e];
                    float v = Elem<VT>::to_f(a.vals[e]);
                    if (j >= a.f) {  // corrupt index: record it and contribute nothing
                        report(a.status, TWELL_ERR_DEVICE_CHECK);
                        j = 0;
                        v = 0.0f;
                    }
                    s_items[buf * kItemCap + fill + i] = make_int2(j, __float_as_int(v));
                }
                fill += take;
                pos += take;
            }
            __syncwarp();
            if (fill >= kItemEager) publish();  // keep the issuer fed from the first rows on
        }
        // end marker, then hand over the last buffer
        if (ok) {
            if (fill == kItemCap) publish();
            if (ok) {
                if (lane == 0) s_items[buf * kItemCap + fill] = make_int2(kEndItem, 0);
                ++fill;
                __syncwarp();
                if (lane == 0) {
                    s_nitems[buf] = fill;
                    mbar_arrive(&lfull[buf]);
                }
            }
        }
    } else if (tid >= C) {
        // ---------------------------------------------------------------- issuer warp (lane 0)
        // Walks the item stream: a row record stages x_r (bulk copy) and its nonzero count into
        // the row ring; a nonzero stages rows j of Wu_s and Wd_s into the slot ring.
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_last();
            const uint64_t pol_x = policy_evict_first();
            int slot = 0, rs = 0, buf = 0;
            uint32_t ph = 0, rph = 0, bph = 0;
            uint32_t issued = 0, issued_ph = 0, xissued = 0, xissued_ph = 0;
            bool ok = true, done = false;
            while (ok && !done) {
                if (!wait_bounded(&lfull[buf], bph, abort_flag, a.status, a.wait_limit_ns)) break;
                const int n = s_nitems[buf];
                for (int i = 0; ok && i < n; ++i) {
                    const int2 it = s_items[buf * kItemCap + i];
                    if (it.x == kEndItem) {
                        done = true;
                        break;
                    }
                    if (it.x < 0) {
                        const int r = ~it.x, nnz = it.y;
                        if (!wait_bounded(&rempty[rs], rph ^ 1u, abort_flag, a.status, a.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
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
                        if (++rs == kRowSlots) {
                            rs = 0;
                            rph ^= 1u;
                        }
                    } else {
                        if (!wait_bounded(&empty[slot], ph ^ 1u, abort_flag, a.status, a.wait_limit_ns)) {
                            ok = false;
                            break;
                        }
                        const size_t j = static_cast<size_t>(it.x);
                        s_a[slot] = __int_as_float(it.y);
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
                mbar_arrive(&lempty[buf]);
                if (++buf == kItemBufs) {
                    buf = 0;
                    bph ^= 1u;
                }
            }
            // no bulk copy may still be writing shared memory when the CTA exits
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s)) wait_bounded(&full[s], (issued_ph >> s) & 1u, nullptr, a.status, a.wait_limit_ns);
            for (int s = 0; s < kRowSlots; ++s)
                if (xissued & (1u << s))
                    wait_bounded(&rfull[s], (xissued_ph >> s) & 1u, nullptr, a.status, a.wait_limit_ns);
        }
    } else {
        // ---------------------------------------------------------------- consumer warps
        // Batch = one nonzero per consumer warp. Warp w forms the whole dot x_r . Wu_s[j] of the
        // batch's w-th nonzero (x_r held in fp32 registers, lane l covering 16-byte chunks
        // l, l+32, ...), reduces it with 5 shuffles and publishes h = a * u; after one named
        // barrier every warp applies all of the batch's rank-1 updates h * Wd_s[j] to its own
        // slice of y_r (lane l of warp w owns chunk 32w + l).
        const int warp = tid >> 5;
        constexpr int YC = XC > 0 ? 1 : 2;  // chunks of y per thread: tid, tid + C
        int slot = 0, rs = 0, buf = 0;
        uint32_t ph = 0, rph = 0;
        for (int r = blockIdx.x; r < a.N; r += gridDim.x) {
            // one lane per warp observes the row record; the named barrier that follows orders the
            // staged x row before every consumer thread's reads
            int rok = 1;
            if (lane == 0) rok = wait_bounded(&rfull[rs], rph, abort_flag, a.status, a.wait_limit_ns) ? 1 : 0;
            if (bar_or(1, C, rok == 0)) break;
            const int nnz = s_nnz[rs];
            float acc[YC][V];
#pragma unroll
            for (int i = 0; i < YC; ++i)
#pragma unroll
                for (int e = 0; e < V; ++e) acc[i][e] = 0.0f;
            float xf[XC > 0 ? XC : 1][V];
            const E* xrow = s_x + static_cast<size_t>(rs) * a.d;
            if (XC > 0 && nnz > 0) {
#pragma unroll
                for (int m = 0; m < (XC > 0 ? XC : 1); ++m) {
                    const int c = lane + 32 * m;
                    if (c < nchunks) unpack16(*reinterpret_cast<const uint4*>(xrow + c * V), xf[m], static_cast<E*>(nullptr));
                    else
#pragma unroll
                        for (int e = 0; e < V; ++e) xf[m][e] = 0.0f;
                }
            }
            bool failed = false;
            for (int b = 0; b < nnz; b += batch) {
                const int nb = min(batch, nnz - b);
                // slot of this warp's nonzero
                int s = slot + warp;
                uint32_t p = ph;
                if (s >= S) {
                    s -= S;
                    p ^= 1u;
                }
                bool okb = true;
                float h = 0.0f;
                if (warp < nb) {
                    int w = 1;
                    if (lane == 0) w = wait_bounded(&full[s], p, abort_flag, a.status, a.wait_limit_ns) ? 1 : 0;
                    okb = __shfl_sync(0xffffffffu, w, 0) != 0;
                    const E* wrow = s_wu + static_cast<size_t>(s) * a.d;
                    float dp[V];
#pragma unroll
                    for (int e = 0; e < V; ++e) dp[e] = 0.0f;
                    if (XC > 0) {
                        uint4 wraw[XC > 0 ? XC : 1];
#pragma unroll
                        for (int m = 0; m < (XC > 0 ? XC : 1); ++m) {
                            const int c = lane + 32 * m;
                            wraw[m] = c < nchunks ? *reinterpret_cast<const uint4*>(wrow + c * V) : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int m = 0; m < (XC > 0 ? XC : 1); ++m) {
                            float wv[V];
                            unpack16(wraw[m], wv, static_cast<E*>(nullptr));
#pragma unroll
                            for (int e = 0; e < V; ++e) dp[e] = fmaf(xf[m][e], wv[e], dp[e]);
                        }
                    } else {
                        for (int c = lane; c < nchunks; c += 32) {
                            float xv[V], wv[V];
                            unpack16(*reinterpret_cast<const uint4*>(xrow + c * V), xv, static_cast<E*>(nullptr));
                            unpack16(*reinterpret_cast<const uint4*>(wrow + c * V), wv, static_cast<E*>(nullptr));
#pragma unroll
                            for (int e = 0; e < V; ++e) dp[e] = fmaf(xv[e], wv[e], dp[e]);
                        }
                    }
                    float dsum = 0.0f;
#pragma unroll
                    for (int e = 0; e < V; ++e) dsum += dp[e];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
                    h = s_a[s] * dsum;
                    if (lane == 0) s_red[buf * (kMaxConsumers / 32) + warp] = h;
                }
                if (bar_or(1, C, !okb)) {
                    failed = true;
                    break;
                }
                // rank-1 updates of this thread's chunk of y_r. Every slot of the batch was observed
                // complete by its dot warp before the named barrier above, which orders the
                // bulk-copied bytes before these reads; the batch's Wd chunks are loaded in groups
                // of four so the shared-memory latencies overlap.
                {
                    const float* hb = s_red + buf * (kMaxConsumers / 32);
#pragma unroll
                    for (int i = 0; i < YC; ++i) {
                        const int q = tid + i * C;
                        if (q >= nchunks) continue;
                        for (int k0 = 0; k0 < nb; k0 += 4) {
                            uint4 w4[4];
                            float h4[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                int sk = slot + k0 + u;
                                if (sk >= S) sk -= S;
                                const bool live = k0 + u < nb;
                                h4[u] = live ? hb[k0 + u] : 0.0f;
                                w4[u] = live ? *reinterpret_cast<const uint4*>(s_wd + static_cast<size_t>(sk) * a.d + q * V)
                                             : make_uint4(0, 0, 0, 0);
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                float wv[V];
                                unpack16(w4[u], wv, static_cast<E*>(nullptr));
#pragma unroll
                                for (int e = 0; e < V; ++e) acc[i][e] = fmaf(h4[u], wv[e], acc[i][e]);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    int sk = slot;
                    for (int k = 0; k < nb; ++k) {
                        mbar_arrive(&empty[sk]);
                        if (++sk == S) sk = 0;
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
            for (int i = 0; i < YC; ++i) {
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

template <typename E, typename VT, int XC>
static twell_status launch_fused(FusedArgs<E, VT> a, cudaStream_t s)
{
    twell_host::DevInfo di;
    if (twell_host::dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    constexpr int V = Elem<E>::kPer16B;
    const int nchunks = a.d / V;
    a.consumers = XC > 0 ? (nchunks + 31) / 32 * 32 : ((nchunks + 1) / 2 + 31) / 32 * 32;
    const int row_bytes = a.d * static_cast<int>(sizeof(E));
    const size_t fixed = FusedLayout(0, row_bytes).total;
    const size_t budget = di.max_smem_optin;
    if (budget <= fixed) return TWELL_ERR_UNSUPPORTED;
    int S = static_cast<int>((budget - fixed) / (2 * static_cast<size_t>(row_bytes)));
    if (S > kMaxSlots) S = kMaxSlots;
    if (S < 4) return TWELL_ERR_UNSUPPORTED;
    a.S = S;
    a.wait_limit_ns = twell_host::wait_limit_ns();
    const FusedLayout layout(S, row_bytes);
    if (row_bytes % 16 != 0 || !layout.aligned()) return TWELL_ERR_UNSUPPORTED;
    const size_t smem = layout.total;
    auto kern = ffn_fused_kernel<E, VT, XC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return TWELL_ERR_CUDA;
    const int grid = a.N < di.sm_count ? a.N : di.sm_count;
    kern<<<grid, a.consumers + 64, smem, s>>>(a);
    return twell_host::launch_status();
}

template <typename E, typename VT>
static twell_status run_fused(const FusedArgs<E, VT>& a, cudaStream_t s)
{
    constexpr int V = Elem<E>::kPer16B;
    const int nchunks = a.d / V;
    if (nchunks <= 32 * 4) return launch_fused<E, VT, 4>(a, s);
    if (nchunks <= 32 * 8) return launch_fused<E, VT, 8>(a, s);
    if (nchunks <= 32 * 10) return launch_fused<E, VT, 10>(a, s);
    if (nchunks <= 2 * kMaxConsumers) return launch_fused<E, VT, 0>(a, s);
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
