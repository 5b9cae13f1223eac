// twell_ffn.cu -- fused up+down projection over a TwELL matrix of gate activations.
//
// For every token row r the kernel walks only the packed nonzeros (column j, value a) of that
// row, gathers row j of Wu_s and row j of Wd_s, forms u = x_r . Wu_s[j], h = a * u and
// accumulates y_r += h * Wd_s[j] in fp32 registers; the hidden activation never leaves the SM
// ([AIM] ¶3; [TG] "Инференс"; [PUL] ¶3; [TC] §2).
//
// GB300 layout. The work is a gather of 2 * d_model * sizeof(E) bytes per nonzero out of weight
// rows that stay resident in the 129 MB L2, plus ~2 * d_model multiply-adds per nonzero. What
// there is to engineer is keeping enough bytes in flight per SM while spending few instructions
// per nonzero. Three kernels share the row stream (RowStream below): one token row is owned by a
// group of G warps; the TwELL metadata runs one 32-nonzero segment ahead: counts of the next row
// are loaded a row ahead, scanned into per-tile offsets in shared memory, and one lane per nonzero
// finds its tile by binary search and loads its index and value into registers. With G = 1 warps
// take rows from a ticket counter (the caller's workspace, cleared on the launch stream), so
// per-token nonzero counts do not unbalance the SMs; groups of G > 1 warps take rows round-robin.
//
// ffn_bulk_kernel (bf16, d_model 512 .. 2048 in steps of 256, 2560 and 3072): lane 0
// of each warp copies whole weight rows into a shared-memory ring with 1-D bulk copies (see the
// kernel); both projections run on the tensor cores (mma.sync) from ldmatrix fragments. Measured
// on the 2048-wide layer: 0.189-0.209 ms, against 0.276 ms for ffn_mma_kernel.
//
// ffn_mma_kernel (bf16, d_model 512, 1024, 1280, 1536 or 2048, where the bulk kernel's ring does
// not fit in shared memory, i.e. very many column tiles): nonzeros are taken in batches of up to
// 16 of one row. The 16 dot products x_r . Wu_s[j] of a batch run on the tensor cores as
// mma.sync m16n8k16 with the batch's weight rows as the 16 rows of A and x_r in every column of
// B (the products need no bf16 -> fp32 conversion; the k order inside a 16-wide block is
// permuted the same way on both sides, so that each lane reads 32 contiguous bytes). The
// rank-1 updates y_r += h * Wd_s[j] run as packed fp32 FMAs on each lane's columns. Weight
// rows move in 4 KB steps (32 bytes per lane per load, so four lanes cover a 128-byte line)
// through a register ring, two or three steps ahead of use across batch and row boundaries.
//
// ffn_rows_kernel (every other shape, fp32): one nonzero at a time, the dot product as a warp
// reduction (plus a named-barrier exchange between the G warps of a row), weight rows of the
// next nonzero loaded while the current one is used.
//
// The bulk kernel's mbarrier waits are bounded (TWELL_ERR_TIMEOUT); the other kernels have no
// spin-wait. The TwELL is checked on the way in (a count above the tile
// width, an in-tile index at or beyond T, a column at or beyond d_ff): a bad entry is recorded
// in the status word as TWELL_ERR_DEVICE_CHECK and contributes nothing, and every access stays
// inside the TwELL's own arrays.
#include "twell_common.cuh"
#include <cuda_fp16.h>

#include "twell_mma.cuh"

namespace twell {

constexpr int kSeg = 32;        // nonzeros per metadata segment (one per lane)
constexpr int kXBufs = 3;       // x_r buffers per warp
constexpr int kCntRegs = 4;     // rows with nt <= 128 tiles get their counts prefetched in registers
constexpr int kMaxTiles = 1024;
constexpr int kCtaWarps = 4;
constexpr int kCtaThreads = 32 * kCtaWarps;
constexpr int kFirst = 1, kLast = 2;

struct __align__(16) SplitItem {
    int row, beg, end, h;  // nonzeros [beg, end) of row; h: the row's first item (kSkipPart: empty)
};
struct __align__(16) HeavyRow {
    int row, nseg, base, done;  // done: items finished so far (zeroed by the plan)
};

template <typename E>
struct RowArgs {
    const E* x;
    const E* Wu;
    const E* Wd;
    const void* vals;  // fp32 or bf16 (vals_bf16)
    const uint8_t* idx;
    const uint16_t* cnt;
    E* y;
    int* tickets;  // G == 1: work counter, zero at launch; with split: [1] items, [2..4] row classes
    int32_t* status;
    int N, d, f, T, nt, nchunks, vals_bf16;
    uint64_t wait_ns;  // bound of every mbarrier wait (ffn_bulk_kernel)
    // Long-row splitting (ffn_bulk_kernel only, split != 0; see split_plan_kernel)
    int split = 0;
    int item_cap = 0;
    const int* list = nullptr;         // [3, N] unsplit rows by class (longest first)
    const SplitItem* items = nullptr;  // [item_cap]
    HeavyRow* heavy = nullptr;         // [item_cap], indexed by a split row's first item
    float* part = nullptr;             // [item_cap, d] fp32 partial y_r of each item
    int f16down = 0;                   // Wd holds fp16 bits (ffn_bulk_kernel only)
};

// Rows with more than `seg` nonzeros are cut into ceil(nnz / seg) items of near-equal length,
// handed out before whole rows; the item that finishes last sums the items' fp32 partial rows in
// item order and stores y_r (so y does not depend on which warp ran what). Whole rows follow in
// three classes, longest first: more than kClassA nonzeros, more than kClassB, the rest. Per-token
// nonzero counts vary by two orders of magnitude ([TC] §3): one warp walking a row of a thousand
// nonzeros would otherwise finish long after all the others. seg is kSplitSeg for large batches
// and shrinks with N down to kSplitSegMin, so that a small batch (decoding a few tokens) spreads
// each row's nonzeros over many warps instead of leaving all but N of them idle.
constexpr int kSplitSeg = 128;
constexpr int kSplitSegMin = 4;
constexpr int kClassA = 64;
constexpr int kClassB = 32;
constexpr int kSkipPart = -2;  // an item left over when the item list ran out of room: no work
constexpr int kWholeRow = -1;  // c_part of a whole row

// Workspace of twell_ffn_fused_fwd (byte offsets, 256-byte aligned): a 256-byte header (work
// counter and the plan's counts), the row lists, the items, the split rows, the partials.
struct FusedWs {
    int item_cap = 0;
    size_t list = 0, items = 0, heavy = 0, part = 0, total = 0;
    __host__ __device__ static size_t up(size_t v) { return (v + 255) & ~size_t(255); }
    // Item slots: N/8 within [4096, 16384] (so that a small batch cut into short items rarely runs
    // out, which would make the split depend on scheduling), and no more than a batch can use.
    __host__ __device__ FusedWs(int N, int d, int f)
    {
        const long long most = static_cast<long long>(N) * ((f + kSplitSegMin - 1) / kSplitSegMin);
        long long c = N / 8;
        c = c < 4096 ? 4096 : (c > 16384 ? 16384 : c);
        if (c > most) c = most;
        item_cap = static_cast<int>(c < 64 ? 64 : c);
        list = 256;
        items = list + up(static_cast<size_t>(N) * 12);
        heavy = items + up(static_cast<size_t>(item_cap) * 16);
        part = heavy + up(static_cast<size_t>(item_cap) * 16);
        total = part + up(static_cast<size_t>(item_cap) * d * 4);
    }
};

__host__ __device__ inline size_t pref_bytes(int nt) { return (static_cast<size_t>(nt + 1) * 4 + 15) & ~size_t(15); }

// ---- packed fp32 pairs (fma.rn.f32x2)

__device__ __forceinline__ uint64_t f2pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t a, uint64_t b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
// Two bf16 in one 32-bit word -> the fp32 pair (low element first). Exact.
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(w << 16), "r"(w & 0xffff0000u));
    return r;
}

// A 16-byte chunk as P fp32 pairs, in element order.
template <typename E>
struct Chunk;
template <>
struct Chunk<__nv_bfloat16> {
    static constexpr int P = 4;
    __device__ __forceinline__ static void pairs(const uint4& v, uint64_t (&o)[4])
    {
        o[0] = bf2_to_f2(v.x);
        o[1] = bf2_to_f2(v.y);
        o[2] = bf2_to_f2(v.z);
        o[3] = bf2_to_f2(v.w);
    }
};
template <>
struct Chunk<float> {
    static constexpr int P = 2;
    __device__ __forceinline__ static void pairs(const uint4& v, uint64_t (&o)[2])
    {
        o[0] = (static_cast<uint64_t>(v.y) << 32) | v.x;
        o[1] = (static_cast<uint64_t>(v.w) << 32) | v.z;
    }
};

// Weight loads: read-only, not kept in L1 (a row is used once per visit), kept in L2.
__device__ __forceinline__ uint4 ldg_keep16(const void* p, uint64_t policy)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(policy));
    return v;
}
// 32 bytes (32-byte aligned) into eight registers.
__device__ __forceinline__ void ldg_keep32(uint32_t (&r)[8], const void* p, uint64_t policy)
{
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "l"(p), "l"(policy));
}

// cp.async: 16-byte global -> shared copies, tracked per thread in commit groups.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bar_sync_named(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}


// Shared memory of one group of G warps: two ticket mailboxes, then the 2 x G partial dot
// products of the general kernel (G <= 4).
constexpr int kGroupBytes = 16 + 2 * 4 * 4;

// ------------------------------------------------------------------------------------------
// The row stream of one group of G warps: row tickets, TwELL metadata one segment ahead, x_r
// staged by cp.async (CPLX 16-byte chunks per lane: chunk q = q0 + m*32*G sits at
// s_x[(xs*CPLX + m)*32 + lane], so with G = 1 a buffer holds x_r contiguously). Every warp of a
// group runs its own copy of the stream over the same rows; the group's first warp takes the row
// tickets and hands them to the others through a mailbox behind the group's named barrier.
template <typename E, int CPLX, int G>
struct RowStream {
    static constexpr int V = Elem<E>::kPer16B;
    uint4* s_x;
    int* s_pref;
    int* s_tk;
    int lane, wg, q0, bar_id, tpar;
    bool pre;
    int tk;
    int creg[kCntRegs];
    int i_row, n_row, i_nnz, i_base, xs_next;              // metadata side
    int nx_row, nx_n, nx_flags, nx_xs, nx_toff;            // next segment (warp-uniform)
    uint32_t nx_idx, nx_val;                               // next segment (one nonzero per lane)
    int c_row, c_n, c_flags, c_xs, c_j, pos;               // current segment
    float c_a;
    int n_beg, n_end, n_part;  // next work item: nonzeros [n_beg, n_end) of n_row; its partial slot
    int i_beg, i_part;         // the item being issued
    int nx_part, c_part;       // partial slot of the next / current segment (kWholeRow: a whole row)
    int s_items, s_cls[3];     // split mode: the plan's items and unsplit rows per class
    int p_kind, p_t;           // lane 0, split mode: the ticket taken one advance ago and its entry,
    int4 p_raw;                // loaded but not yet used (1: item, 2: list row, 3: past the end)

    __device__ void next_ticket(const RowArgs<E>& a)
    {
        tk = 0;
        if (wg == 0 && lane == 0) tk = atomicAdd(a.tickets, 1);
    }
    // The ticket taken one call of next_ticket earlier (its atomic has had a row's time to land).
    __device__ int ticket_row()
    {
        if constexpr (G == 1) {
            return __shfl_sync(0xffffffffu, tk, 0);
        } else {
            int v = 0;
            if (wg == 0) {
                v = __shfl_sync(0xffffffffu, tk, 0);
                if (lane == 0) s_tk[tpar] = v;
            }
            bar_sync_named(bar_id, 32 * G);
            if (wg != 0) v = s_tk[tpar];
            tpar ^= 1;  // the next write goes to the other box: a reader may still be on this one
            return v;
        }
    }
    __device__ void load_counts(const RowArgs<E>& a, int r)
    {
#pragma unroll
        for (int m = 0; m < kCntRegs; ++m) {
            const int t = lane + 32 * m;
            creg[m] = (pre && r < a.N && t < a.nt) ? static_cast<int>(a.cnt[static_cast<size_t>(r) * a.nt + t]) : 0;
        }
    }
    // exclusive offsets of row r's tiles into s_pref[0..nt]; returns the row's nonzeros
    __device__ int scan_row(const RowArgs<E>& a, int r)
    {
        __syncwarp();  // every lane is done reading the previous row's offsets
        int run = 0;
        const int iters = (a.nt + 31) / 32;
        for (int m = 0; m < iters; ++m) {
            const int t = lane + 32 * m;
            int v = 0;
            if (pre) {
#pragma unroll
                for (int mm = 0; mm < kCntRegs; ++mm)
                    if (mm == m) v = creg[mm];
            } else if (t < a.nt) {
                v = a.cnt[static_cast<size_t>(r) * a.nt + t];
            }
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
        if (lane == 0) s_pref[a.nt] = run;
        __syncwarp();
        return run;
    }
    // Split mode, lane 0: start the load of ticket t's entry (used one advance later).
    __device__ void fetch(const RowArgs<E>& a, int t)
    {
        p_t = t;
        if (t < s_items) {
            p_kind = 1;
            p_raw = *reinterpret_cast<const int4*>(a.items + t);
            return;
        }
        int i = t - s_items;
        p_kind = 3;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            if (p_kind == 3 && i < s_cls[k]) {
                p_kind = 2;
                p_raw.x = a.list[static_cast<size_t>(k) * a.N + i];
            }
            i -= s_cls[k];
        }
    }
    // Split mode: the next work item from the entry fetched one advance ago; fetch the entry of the
    // ticket taken one advance ago; take a new ticket.
    __device__ void next_item(const RowArgs<E>& a)
    {
        int r = a.N, b = 0, e = 0, pp = kWholeRow;
        if (lane == 0) {
            if (p_kind == 1) {
                if (p_raw.w == kSkipPart) {
                    r = 0;
                    pp = kSkipPart;
                } else {
                    r = p_raw.x;
                    b = p_raw.y;
                    e = p_raw.z;
                    pp = p_t;
                }
            } else if (p_kind == 2) {
                r = p_raw.x;
                e = 0x7fffffff;
            }
            fetch(a, tk);
        }
        n_row = __shfl_sync(0xffffffffu, r, 0);
        n_beg = __shfl_sync(0xffffffffu, b, 0);
        n_end = __shfl_sync(0xffffffffu, e, 0);
        n_part = __shfl_sync(0xffffffffu, pp, 0);
        load_counts(a, n_row);
        next_ticket(a);
    }
    __device__ void advance_issue_row(const RowArgs<E>& a)
    {
        i_row = n_row;
        i_part = n_part;
        const int tot = i_row < a.N ? scan_row(a, i_row) : 0;
        i_nnz = min(n_end, tot);
        i_beg = min(n_beg, i_nnz);
        i_base = i_beg;
        if (a.split) {
            next_item(a);
        } else {
            n_row = ticket_row();
            load_counts(a, n_row);
            next_ticket(a);
        }
    }
    // Describe the next segment (loads of its indices and values stay in flight) and, at a row
    // start, copy x of that row into the next x buffer. Commits exactly one cp.async group.
    __device__ void issue_segment(const RowArgs<E>& a)
    {
        if (i_row >= a.N) {
            nx_n = -1;  // end of this group's rows
            cp_async_commit();
            return;
        }
        const int n = min(kSeg, i_nnz - i_base);
        nx_row = i_row;
        nx_n = n;
        nx_part = i_part;
        nx_flags = (i_base == i_beg ? kFirst : 0) | (i_base + n >= i_nnz ? kLast : 0);
        if (i_base == i_beg && n > 0) {
            nx_xs = xs_next;
            xs_next = xs_next + 1 == kXBufs ? 0 : xs_next + 1;
            const E* xr = a.x + static_cast<size_t>(i_row) * a.d;
#pragma unroll
            for (int m = 0; m < CPLX; ++m) {
                const int q = q0 + m * 32 * G;
                if (q < a.nchunks) cp_async16(&s_x[(nx_xs * CPLX + m) * 32 + lane], xr + q * V);
            }
        }
        if (lane < n) {
            const int gp = i_base + lane;
            int lo = 0, hi = a.nt;  // s_pref[lo] <= gp < s_pref[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_pref[mid] <= gp) lo = mid;
                else hi = mid;
            }
            const size_t e = (static_cast<size_t>(i_row) * a.nt + lo) * a.T + (gp - s_pref[lo]);
            nx_toff = lo * a.T;
            nx_idx = a.idx[e];
            nx_val = a.vals_bf16 ? static_cast<uint32_t>(static_cast<const uint16_t*>(a.vals)[e]) << 16
                                 : static_cast<const uint32_t*>(a.vals)[e];
        }
        cp_async_commit();
        i_base += n;
        if (nx_flags & kLast) advance_issue_row(a);
    }
    __device__ void take_segment(const RowArgs<E>& a)
    {
        c_row = nx_row;
        c_n = nx_n;
        c_flags = nx_flags;
        c_xs = nx_xs;
        c_part = nx_part;
        if (lane < c_n) {
            int j = nx_toff + static_cast<int>(nx_idx);
            float v = __uint_as_float(nx_val);
            if (static_cast<int>(nx_idx) >= a.T || j >= a.f) {  // corrupt entry: record it, contribute nothing
                report(a.status, TWELL_ERR_DEVICE_CHECK);
                j = 0;
                v = 0.0f;
            }
            c_j = j;
            c_a = v;
        }
    }
    __device__ void zero_row(const RowArgs<E>& a, int row)
    {
        E* yr = a.y + static_cast<size_t>(row) * a.d;
        for (int q = q0; q < a.nchunks; q += 32 * G) st_stream16(yr + q * V, make_uint4(0, 0, 0, 0));
    }
    __device__ void init(const RowArgs<E>& a, uint4* sx, int* spref, int* stk, int lane_, int wg_, int bar)
    {
        s_x = sx;
        s_pref = spref;
        s_tk = stk;
        lane = lane_;
        wg = wg_;
        q0 = wg * 32 + lane;
        bar_id = bar;
        tpar = 0;
        pre = a.nt <= 32 * kCntRegs;
        tk = 0;
        i_row = n_row = a.N;
        i_nnz = i_base = xs_next = 0;
        nx_row = nx_flags = nx_xs = nx_toff = 0;
        nx_n = -1;
        nx_idx = nx_val = 0;
        c_row = c_n = c_flags = c_xs = c_j = pos = 0;
        c_a = 0.0f;
        n_beg = 0;
        n_end = 0x7fffffff;
        n_part = i_beg = i_part = nx_part = c_part = kWholeRow;
        p_kind = 3;
        p_t = 0;
        p_raw = make_int4(0, 0, 0, 0);
        s_items = s_cls[0] = s_cls[1] = s_cls[2] = 0;
        // pipeline fill: first row's counts and offsets, the next row's counts, the first segment
        if (a.split) {  // one stage more: ticket -> item or list entry -> counts -> offsets
            s_items = min(a.tickets[1], a.item_cap);
            s_cls[0] = a.tickets[2];
            s_cls[1] = a.tickets[3];
            s_cls[2] = a.tickets[4];
            next_ticket(a);
            if (lane == 0) fetch(a, tk);
            next_ticket(a);
            next_item(a);
        } else {
            next_ticket(a);
            n_row = ticket_row();
            load_counts(a, n_row);
            next_ticket(a);
        }
        advance_issue_row(a);
        issue_segment(a);
    }
    // Make the current segment one with nonzeros left to take (pos < c_n); false at the end.
    // Rows without nonzeros met on the way get y_r = 0.
    __device__ bool ready(const RowArgs<E>& a)
    {
        while (pos >= c_n) {
            if (c_n < 0) return false;
            take_segment(a);
            issue_segment(a);
            pos = 0;
            if (c_n < 0) return false;
            if (c_n == 0) {
                if (c_part == kWholeRow) zero_row(a, c_row);  // a row without nonzeros
                continue;
            }
            if (c_flags & kFirst) {
                cp_async_wait<1>();  // x of this row: the group before the one just committed
                __syncwarp();        // lanes read chunks other lanes copied
            }
        }
        return true;
    }
};

// ------------------------------------------------------------------------------------------
// General kernel: one nonzero at a time.

struct Entry {
    int j;      // hidden unit
    float a;    // gate activation
    int row;    // token row
    int xs;     // x buffer holding x_row
    int flags;  // kFirst: first nonzero of the row; kLast: last one
};

template <int CPL>
struct RowSmem {
    __host__ __device__ static size_t x_bytes() { return static_cast<size_t>(kXBufs) * CPL * 32 * 16; }
    __host__ __device__ static size_t warp_bytes(int nt) { return x_bytes() + pref_bytes(nt); }
    __host__ __device__ static size_t cta_bytes(int nt) { return kCtaWarps * warp_bytes(nt) + kCtaWarps * kGroupBytes; }
};

template <typename E, int CPL, int G>
__global__ void __launch_bounds__(kCtaThreads, (CPL >= 5 ? 2 : CPL == 4 ? 3 : 4)) ffn_rows_kernel(const RowArgs<E> a)
{
    constexpr int V = Elem<E>::kPer16B;
    constexpr int P = Chunk<E>::P;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wg = warp % G, grp = warp / G;
    const size_t wbytes = RowSmem<CPL>::warp_bytes(a.nt);
    uint4* s_x = reinterpret_cast<uint4*>(smem + warp * wbytes);
    int* s_pref = reinterpret_cast<int*>(smem + warp * wbytes + RowSmem<CPL>::x_bytes());
    uint8_t* gsm = smem + kCtaWarps * wbytes + grp * kGroupBytes;
    int* s_tk = reinterpret_cast<int*>(gsm);
    float* s_part = reinterpret_cast<float*>(gsm + 16);

    const uint64_t pol = policy_evict_last();
    const int nchunks = a.nchunks;
    const int q0 = wg * 32 + lane;  // chunk of m = 0; chunk m is q0 + m * 32 * G

    RowStream<E, CPL, G> rs;
    rs.init(a, s_x, s_pref, s_tk, lane, wg, 1 + grp);
    auto next_entry = [&](Entry& en) -> bool {
        if (!rs.ready(a)) return false;
        en.j = __shfl_sync(0xffffffffu, rs.c_j, rs.pos);
        en.a = __shfl_sync(0xffffffffu, rs.c_a, rs.pos);
        en.row = rs.c_row;
        en.xs = rs.c_xs;
        en.flags = (rs.pos == 0 ? (rs.c_flags & kFirst) : 0) | (rs.pos == rs.c_n - 1 ? (rs.c_flags & kLast) : 0);
        ++rs.pos;
        return true;
    };

    uint64_t acc[CPL][P];
#pragma unroll
    for (int m = 0; m < CPL; ++m)
#pragma unroll
        for (int p = 0; p < P; ++p) acc[m][p] = 0;
    auto store_row = [&](int row) {
        E* yr = a.y + static_cast<size_t>(row) * a.d;
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            const int q = q0 + m * 32 * G;
            if (q >= nchunks) continue;
            float fv[V];
#pragma unroll
            for (int p = 0; p < P; ++p) f2unpack(acc[m][p], fv[2 * p], fv[2 * p + 1]);
            st_stream16(yr + q * V, pack16(fv, static_cast<E*>(nullptr)));
        }
    };

    int par = 0;
    auto load_w = [&](uint4 (&wu)[CPL], uint4 (&wd)[CPL], int j) {
        const E* pu = a.Wu + static_cast<size_t>(j) * a.d;
        const E* pd = a.Wd + static_cast<size_t>(j) * a.d;
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            const int q = q0 + m * 32 * G;
            if (q < nchunks) {
                wu[m] = ldg_keep16(pu + q * V, pol);
                wd[m] = ldg_keep16(pd + q * V, pol);
            }
        }
    };
    auto compute = [&](const uint4 (&wu)[CPL], const uint4 (&wd)[CPL], const Entry& en) {
        if (en.flags & kFirst) {
#pragma unroll
            for (int m = 0; m < CPL; ++m)
#pragma unroll
                for (int p = 0; p < P; ++p) acc[m][p] = 0;
        }
        uint64_t s[P];
#pragma unroll
        for (int p = 0; p < P; ++p) s[p] = 0;
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            const int q = q0 + m * 32 * G;
            if (q < nchunks) {
                uint64_t xp[P], wp[P];
                Chunk<E>::pairs(s_x[(en.xs * CPL + m) * 32 + lane], xp);
                Chunk<E>::pairs(wu[m], wp);
#pragma unroll
                for (int p = 0; p < P; ++p) fma2(s[p], xp[p], wp[p]);
            }
        }
        float part = 0.0f;
#pragma unroll
        for (int p = 0; p < P; ++p) {
            float lo, hi;
            f2unpack(s[p], lo, hi);
            part += lo + hi;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        float u = part;
        if constexpr (G > 1) {
            if (lane == 0) s_part[par * G + wg] = part;
            bar_sync_named(1 + grp, 32 * G);
            u = 0.0f;
#pragma unroll
            for (int g = 0; g < G; ++g) u += s_part[par * G + g];
            par ^= 1;
        }
        const float h = en.a * u;
        const uint64_t h2 = f2pack(h, h);
#pragma unroll
        for (int m = 0; m < CPL; ++m) {
            const int q = q0 + m * 32 * G;
            if (q < nchunks) {
                uint64_t wp[P];
                Chunk<E>::pairs(wd[m], wp);
#pragma unroll
                for (int p = 0; p < P; ++p) fma2(acc[m][p], h2, wp[p]);
            }
        }
        if (en.flags & kLast) store_row(en.row);
    };

    uint4 ua[CPL], da[CPL], ub[CPL], db[CPL];
#pragma unroll
    for (int m = 0; m < CPL; ++m) ua[m] = da[m] = ub[m] = db[m] = make_uint4(0, 0, 0, 0);
    Entry ea, eb;
    bool ha = next_entry(ea);
    if (ha) load_w(ua, da, ea.j);
    while (ha) {
        const bool hb = next_entry(eb);
        if (hb) load_w(ub, db, eb.j);
        compute(ua, da, ea);
        if (!hb) break;
        ha = next_entry(ea);
        if (ha) load_w(ua, da, ea.j);
        compute(ub, db, eb);
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------------------------------
// Tensor-core kernel (bf16, d_model = 256 * CPLX <= 2048): one warp per token row.

constexpr int kBatch = 16;  // nonzeros per batch: the m dimension of m16n8k16
constexpr int kBatchSlots = 4;

struct __align__(16) BatchDesc {
    int row, k, xs, flags;  // flags: kFirst = the row's first batch, kLast = its last
    int j[kBatch];
    float a[kBatch];
    float h[kBatch];        // h = a * u, filled when the batch's dot products are done
};

template <int CPLX>  // 256-column blocks per warp (16-byte x chunks per lane)
struct MmaSmem {
    __host__ __device__ static size_t x_bytes() { return static_cast<size_t>(kXBufs) * CPLX * 32 * 16; }
    __host__ __device__ static size_t warp_bytes(int nt)
    {
        return x_bytes() + pref_bytes(nt) + kBatchSlots * sizeof(BatchDesc);
    }
    __host__ __device__ static size_t cta_bytes(int nt) { return kCtaWarps * (warp_bytes(nt) + kGroupBytes); }
};

// CPLX: 256-column blocks of d_model; R: depth of the register ring of 4 KB steps.
template <int CPLX, int R>
__global__ void __launch_bounds__(kCtaThreads, 2) ffn_mma_kernel(const RowArgs<__nv_bfloat16> a)
{
    constexpr int G = 1;
    using E = __nv_bfloat16;
    constexpr int CPL = (CPLX + 1) / 2;  // 32-byte chunks per lane of y_r in the down projection
    constexpr int N32 = 16 * CPLX;       // 32-byte chunks of a row (lane l owns l, l + 32, ...)
    constexpr int EPS = 4 / CPL;         // nonzeros per down-projection step
    constexpr int nU = 2 * CPLX;         // up-projection steps per batch (128 columns of d_model each)
    constexpr int kU = 1, kD = 2, kEnd = 3;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const size_t wbytes = MmaSmem<CPLX>::warp_bytes(a.nt);
    uint8_t* wsm = smem + warp * wbytes;
    uint4* s_x = reinterpret_cast<uint4*>(wsm);
    int* s_pref = reinterpret_cast<int*>(wsm + MmaSmem<CPLX>::x_bytes());
    BatchDesc* s_bd = reinterpret_cast<BatchDesc*>(wsm + MmaSmem<CPLX>::x_bytes() + pref_bytes(a.nt));
    int* s_tk = reinterpret_cast<int*>(smem + kCtaWarps * wbytes + warp * kGroupBytes);  // unused with G = 1

    const uint64_t pol = policy_evict_last();

    RowStream<E, CPLX, G> rs;
    rs.init(a, s_x, s_pref, s_tk, lane, 0, 1 + warp);

    // -------------------------------------------------------------- issue side: 4 KB steps
    // A batch of k <= 16 nonzeros is nU up-projection steps (step i covers columns 128i + [0, 128):
    // lane (g, t) loads 32 bytes of Wu_s[j_g] and of Wu_s[j_{g+8}] at offset 64c + 16t, c = 0, 1)
    // followed by ceil(k / EPS) down-projection steps (lane loads its CPL 32-byte chunks of
    // Wd_s[j_e] for EPS nonzeros).
    // The tag of a step: kind | batch slot << 2 | step << 4.
    int is_slot = 0, is_step = 0, is_nsteps = 0, is_k = 0, nslot = 0;
    bool ended = false;
    auto form_batch = [&](BatchDesc* D) -> bool {
        if (!rs.ready(a)) return false;
        const int k = min(kBatch, rs.c_n - rs.pos);
        if (lane >= rs.pos && lane < rs.pos + k) {
            D->j[lane - rs.pos] = rs.c_j;
            D->a[lane - rs.pos] = rs.c_a;
        }
        if (lane == 0) {
            D->row = rs.c_row;
            D->k = k;
            D->xs = rs.c_xs;
            D->flags = (rs.pos == 0 ? (rs.c_flags & kFirst) : 0) | (rs.pos + k == rs.c_n ? (rs.c_flags & kLast) : 0);
        }
        __syncwarp();
        rs.pos += k;
        return true;
    };
    auto issue = [&](uint32_t (&B)[4][8], int& tag) {
        if (ended) {
            tag = kEnd;
            return;
        }
        if (is_step == is_nsteps) {
            if (!form_batch(&s_bd[nslot])) {
                ended = true;
                tag = kEnd;
                return;
            }
            is_slot = nslot;
            nslot = (nslot + 1) & (kBatchSlots - 1);
            is_k = s_bd[is_slot].k;
            is_nsteps = nU + (is_k + EPS - 1) / EPS;
            is_step = 0;
        }
        const BatchDesc* D = &s_bd[is_slot];
        if (is_step < nU) {
            const int col = 128 * is_step + 16 * t;
            if (g < is_k) {
                const E* w = a.Wu + static_cast<size_t>(D->j[g]) * a.d + col;
                ldg_keep32(B[0], w, pol);
                ldg_keep32(B[2], w + 64, pol);
            }
            if (g + 8 < is_k) {
                const E* w = a.Wu + static_cast<size_t>(D->j[g + 8]) * a.d + col;
                ldg_keep32(B[1], w, pol);
                ldg_keep32(B[3], w + 64, pol);
            }
            tag = kU;
        } else {
            const int e0 = (is_step - nU) * EPS;
#pragma unroll
            for (int ee = 0; ee < EPS; ++ee) {
                if (e0 + ee < is_k) {
                    const E* w = a.Wd + static_cast<size_t>(D->j[e0 + ee]) * a.d + 16 * lane;
#pragma unroll
                    for (int m = 0; m < CPL; ++m)
                        if (lane + 32 * m < N32) ldg_keep32(B[ee * CPL + m], w + 512 * m, pol);
                }
            }
            tag = kD;
        }
        tag |= (is_slot << 2) | (is_step << 4);
        ++is_step;
    };

    // -------------------------------------------------------------- process side
    float macc[4][4];  // four accumulator sets: independent mma chains
#pragma unroll
    for (int i = 0; i < 4; ++i) macc[i][0] = macc[i][1] = macc[i][2] = macc[i][3] = 0.0f;
    uint64_t acc[CPL][8];
#pragma unroll
    for (int m = 0; m < CPL; ++m)
#pragma unroll
        for (int w = 0; w < 8; ++w) acc[m][w] = 0;
    auto process = [&](const uint32_t (&B)[4][8], int tag) {
        BatchDesc* D = &s_bd[(tag >> 2) & (kBatchSlots - 1)];
        const int step = tag >> 4;
        if ((tag & 3) == kU) {
            if (step == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) macc[i][0] = macc[i][1] = macc[i][2] = macc[i][3] = 0.0f;
            }
            // A row m is the batch's nonzero m (rows g: B[0], B[2]; rows g+8: B[1], B[3]); x_r in
            // every column of B. Inside each 16-wide k block, k slots (2t, 2t+1, 2t+8, 2t+9) hold
            // columns o+4b .. o+4b+3 of the step's 128 columns with o = 64c + 16t, on both sides.
            const uint4* xr = s_x + (D->xs * CPLX + (step >> 1)) * 32 + 16 * (step & 1);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const uint32_t(&Wg)[8] = B[2 * cc];
                const uint32_t(&Wg8)[8] = B[2 * cc + 1];
                const uint4 X0 = xr[8 * cc + 2 * t], X1 = xr[8 * cc + 2 * t + 1];
                mma_bf16(macc[0], Wg[0], Wg8[0], Wg[1], Wg8[1], X0.x, X0.y);
                mma_bf16(macc[1], Wg[2], Wg8[2], Wg[3], Wg8[3], X0.z, X0.w);
                mma_bf16(macc[2], Wg[4], Wg8[4], Wg[5], Wg8[5], X1.x, X1.y);
                mma_bf16(macc[3], Wg[6], Wg8[6], Wg[7], Wg8[7], X1.z, X1.w);
            }
            if (step == nU - 1) {
                // lane (g, t) holds u of nonzeros g (D row g) and g+8 (row g+8), the same in every
                // column of D
                const float u0 = (macc[0][0] + macc[1][0]) + (macc[2][0] + macc[3][0]);
                const float u1 = (macc[0][2] + macc[1][2]) + (macc[2][2] + macc[3][2]);
                if (t == 0) {
                    D->h[g] = D->a[g] * u0;
                    D->h[g + 8] = D->a[g + 8] * u1;
                }
                __syncwarp();
            }
        } else {
            const int e0 = (step - nU) * EPS;
#pragma unroll
            for (int ee = 0; ee < EPS; ++ee) {
                if (e0 + ee < D->k) {
                    const float h = D->h[e0 + ee];
                    const uint64_t h2 = f2pack(h, h);
#pragma unroll
                    for (int m = 0; m < CPL; ++m)
                        if (lane + 32 * m < N32) {
#pragma unroll
                            for (int w = 0; w < 8; ++w) fma2(acc[m][w], h2, bf2_to_f2(B[ee * CPL + m][w]));
                        }
                }
            }
            if (e0 + EPS >= D->k && (D->flags & kLast)) {
                E* yr = a.y + static_cast<size_t>(D->row) * a.d + 16 * lane;
#pragma unroll
                for (int m = 0; m < CPL; ++m) {
                    float lo8[8], hi8[8];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        f2unpack(acc[m][w], lo8[2 * w], lo8[2 * w + 1]);
                        f2unpack(acc[m][w + 4], hi8[2 * w], hi8[2 * w + 1]);
                    }
                    if (lane + 32 * m < N32) {
                        st_stream16(yr + 512 * m, pack16(lo8, static_cast<E*>(nullptr)));
                        st_stream16(yr + 512 * m + 8, pack16(hi8, static_cast<E*>(nullptr)));
                    }
#pragma unroll
                    for (int w = 0; w < 8; ++w) acc[m][w] = 0;
                }
            }
        }
    };

    uint32_t B[R][4][8];
    int tg[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int w = 0; w < 8; ++w) B[r][i][w] = 0;
#pragma unroll
    for (int r = 0; r < R - 1; ++r) issue(B[r], tg[r]);
    bool run = true;
    while (run) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (run) {
                issue(B[(r + R - 1) % R], tg[(r + R - 1) % R]);
                if (tg[r] == kEnd) run = false;
                else process(B[r], tg[r]);
            }
        }
    }
    cp_async_wait<0>();
}


// ------------------------------------------------------------------------------------------
// Bulk-copy tensor-core kernel (bf16, d_model = 256 * NS): one warp per token row.
//
// Staging. Lane 0 of every warp copies, per nonzero, the whole rows Wu_s[j] and Wd_s[j] (and x_r
// at the row's first nonzero) into one slot of the warp's S-slot ring in shared memory with 1-D
// bulk copies (cp.async.bulk) that complete on the slot's mbarrier, S - 1 nonzeros ahead of use
// and across row boundaries. Many warps issuing such copies reach ~20 TB/s of random 4 KB rows out
// of L2, and the bytes in flight cost no registers.
//
// Both projections run as mma.sync m16n8k16 on operands read with ldmatrix.trans. Chunk c is
// columns [128c, 128c + 128) of d_model, with X[k][m] = x_r[128c + 8k + m] and
// W[k][n] = row[128c + 8k + n] (k < 16; m, n < 8):
//   up:   A = X^T in rows 0..7 (rows 8..15 unused), B = Wu_s[j] chunk, so D[m][m] = sum_k X[k][m] W[k][m]
//         and the trace of D summed over the chunks is u = x_r . Wu_s[j]; the diagonal sits in the
//         eight lanes (g, t) with g >> 1 = t, which sum it in three xor steps (4, 9, 18) that stay
//         among them;
//   down: A = h * I (only those eight lanes hold its diagonal), B = Wd_s[j] chunk, so D += h * W:
//         the 16 x 8 accumulator of chunk c holds y_r[128c + 8m + n] in fp32, in pairs of adjacent
//         columns per lane, and y_r is stored straight from it. h is fp32 and the operands bf16, so
//         h goes in as two MMAs, with hi = bf16(h) and lo = bf16(h - hi) (h to ~16 bits).
template <int NS>
struct BulkLayout {
    static constexpr uint32_t kRow = 512u * NS;  // bytes of one bf16 row of d_model
    static constexpr uint32_t kSlot = 3 * kRow;   // Wu_s[j], Wd_s[j], x_r (row starts only)
    __host__ __device__ static size_t warp_bytes(int S, int nt)
    {
        return (static_cast<size_t>(S) * (kSlot + 16 + 8) + pref_bytes(nt) + 127) & ~size_t(127);
    }
};
struct __align__(16) SlotDesc {
    int row, flags;
    float a;
    int part;  // partial slot of a split row's item, kWholeRow for a whole row
};


// NS: 256-column spans of d_model; S: ring slots per warp; WPC: warps per CTA. F16DOWN: Wd_s holds
// fp16 bits and the down projection is one fp16 product per chunk, with h rounded once to fp16
// (11 significant bits), instead of two bf16 products with h as a bf16 hi + lo pair.
template <int NS, int S, int WPC, bool F16DOWN = false>
__global__ void __launch_bounds__(32 * WPC, 1) ffn_bulk_kernel(const RowArgs<__nv_bfloat16> a)
{
    using E = __nv_bfloat16;
    using L = BulkLayout<NS>;
    constexpr int NC = 2 * NS;  // 128-column chunks
    static_assert(NC >= 4, "four accumulator chains in the up projection");
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    uint8_t* wbase = smem + warp * L::warp_bytes(S, a.nt);
    SlotDesc* desc = reinterpret_cast<SlotDesc*>(wbase + S * L::kSlot);
    uint64_t* bar = reinterpret_cast<uint64_t*>(desc + S);
    int* s_pref = reinterpret_cast<int*>(bar + S);
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const uint64_t pol_w = policy_evict_last(), pol_x = policy_evict_first();
    // launched as a programmatic dependent of the plan kernel: its items, lists and counts (and the
    // work counter cleared before it) are visible once that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    RowStream<E, 0, 1> rs;
    rs.init(a, nullptr, s_pref, nullptr, lane, 0, 0);

    // -------------------------------------------------------------- issue: one nonzero per slot
    int n_issued = 0;
    bool ended = false;
    auto issue = [&]() {
        if (ended) return;
        if (!rs.ready(a)) {
            ended = true;
            return;
        }
        const int p = rs.pos;
        const int j = __shfl_sync(0xffffffffu, rs.c_j, p);
        const float av = __shfl_sync(0xffffffffu, rs.c_a, p);
        const int flags = (p == 0 ? (rs.c_flags & kFirst) : 0) | (p == rs.c_n - 1 ? (rs.c_flags & kLast) : 0);
        ++rs.pos;
        const int s = n_issued % S;
        if (lane == 0) {
            desc[s] = SlotDesc{rs.c_row, flags, av, rs.c_part};
            uint8_t* slot = wbase + s * L::kSlot;
            mbar_arrive_expect_tx(&bar[s], (flags & kFirst) ? 3 * L::kRow : 2 * L::kRow);
            bulk_load(slot, a.Wu + static_cast<size_t>(j) * a.d, L::kRow, &bar[s], pol_w);
            bulk_load(slot + L::kRow, a.Wd + static_cast<size_t>(j) * a.d, L::kRow, &bar[s], pol_w);
            if (flags & kFirst)
                bulk_load(slot + 2 * L::kRow, a.x + static_cast<size_t>(rs.c_row) * a.d, L::kRow, &bar[s], pol_x);
        }
        ++n_issued;
    };

    // -------------------------------------------------------------- compute
    const bool diag = (g >> 1) == t;  // this lane holds the diagonal element g & 1 of its pairs
    const uint32_t hmask = diag ? ((g & 1) ? 0xFFFF0000u : 0x0000FFFFu) : 0u;
    // x_r as the A operands of the up projection, one register quad per chunk: a0 and a2 are the
    // chunk's X^T blocks, a1 and a3 (rows 8..15 of A, whose products are never read) the
    // neighbouring chunk's, so one ldmatrix yields a whole operand. Lane offsets into a 512-byte
    // span for the quad of its even chunk (order: even lo, odd lo, even hi, odd hi) and odd chunk.
    const int mi = lane >> 3, mr = lane & 7;
    const uint32_t xoff_e = 16u * mr + ((mi & 1) ? 256u : 0u) + ((mi & 2) ? 128u : 0u);
    const uint32_t xoff_o = 16u * mr + ((mi & 1) ? 0u : 256u) + ((mi & 2) ? 128u : 0u);
    uint32_t xq[NC][4];
    float yacc[NC][4];  // y_r: chunk c, columns 128c + 8g + 2t (+1) and 128c + 64 + 8g + 2t (+1)
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        xq[c][0] = xq[c][1] = xq[c][2] = xq[c][3] = 0u;
        yacc[c][0] = yacc[c][1] = yacc[c][2] = yacc[c][3] = 0.0f;
    }
    // y_r out of the accumulators (bf16 pairs), which are cleared for the next row
    auto store_y = [&](int row) {
        uint32_t* yr = reinterpret_cast<uint32_t*>(a.y + static_cast<size_t>(row) * a.d) + 4 * g + t;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            yr[64 * c] = bf16x2_rn(yacc[c][0], yacc[c][1]);
            yr[64 * c + 32] = bf16x2_rn(yacc[c][2], yacc[c][3]);
            yacc[c][0] = yacc[c][1] = yacc[c][2] = yacc[c][3] = 0.0f;
        }
    };
    for (int i = 0; i < S; ++i) issue();
    __syncwarp();
    int n_done = 0;
    while (n_done < n_issued) {
        const int s = n_done % S;
        const bool ok =
            __all_sync(0xffffffffu, wait_bounded<false, 20000>(&bar[s], static_cast<uint32_t>(n_done / S) & 1u,
                                                              nullptr, a.status, a.wait_ns));
        if (!ok) break;
        const SlotDesc D = desc[s];
        const uint32_t sb = smem_u32(wbase + s * L::kSlot);
        const uint32_t su = sb + 16u * lane;
        if (D.flags & kFirst) {
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                ldsm_x4_trans(xq[2 * q], sb + 2 * L::kRow + 512u * q + xoff_e);
                ldsm_x4_trans(xq[2 * q + 1], sb + 2 * L::kRow + 512u * q + xoff_o);
            }
        }
        // up projection: four independent accumulator chains
        float uc[4][4];
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            uint32_t w[4];
            ldsm_x4_trans(w, su + 512u * q);
            const uint32_t(&e)[4] = xq[2 * q];
            const uint32_t(&o)[4] = xq[2 * q + 1];
            if (q < 2) {
                mma_bf16_first(uc[2 * q], e[0], e[1], e[2], e[3], w[0], w[1]);
                mma_bf16_first(uc[2 * q + 1], o[0], o[1], o[2], o[3], w[2], w[3]);
            } else {
                mma_bf16(uc[(2 * q) & 3], e[0], e[1], e[2], e[3], w[0], w[1]);
                mma_bf16(uc[(2 * q + 1) & 3], o[0], o[1], o[2], o[3], w[2], w[3]);
            }
        }
        const float s0 = (uc[0][0] + uc[1][0]) + (uc[2][0] + uc[3][0]);
        const float s1 = (uc[0][1] + uc[1][1]) + (uc[2][1] + uc[3][1]);
        float u = diag ? ((g & 1) ? s1 : s0) : 0.0f;
        u += __shfl_xor_sync(0xffffffffu, u, 4);
        u += __shfl_xor_sync(0xffffffffu, u, 9);
        u += __shfl_xor_sync(0xffffffffu, u, 18);
        const float h = D.a * u;
        if constexpr (F16DOWN) {
            // down projection y_r += h * Wd_s[j], h and the row in fp16
            const uint32_t hd = f16x2_rn(h, h) & hmask;
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                uint32_t w[4];
                ldsm_x4_trans(w, su + L::kRow + 512u * q);
                mma_f16(yacc[2 * q], hd, 0u, 0u, hd, w[0], w[1]);
                mma_f16(yacc[2 * q + 1], hd, 0u, 0u, hd, w[2], w[3]);
            }
        } else {
            // h = hi + lo, both bf16: the pair carries h to ~16 significant bits
            const uint32_t hi2 = bf16x2_rn(h, h);
            const float lo = h - __uint_as_float(hi2 << 16);
            const uint32_t hd = hi2 & hmask, ld = bf16x2_rn(lo, lo) & hmask;
            // down projection: y_r += h * Wd_s[j]
#pragma unroll
            for (int q = 0; q < NS; ++q) {
                uint32_t w[4];
                ldsm_x4_trans(w, su + L::kRow + 512u * q);
                mma_bf16(yacc[2 * q], hd, 0u, 0u, hd, w[0], w[1]);
                mma_bf16(yacc[2 * q + 1], hd, 0u, 0u, hd, w[2], w[3]);
                mma_bf16(yacc[2 * q], ld, 0u, 0u, ld, w[0], w[1]);
                mma_bf16(yacc[2 * q + 1], ld, 0u, 0u, ld, w[2], w[3]);
            }
        }
        if (D.flags & kLast) {
            if (D.part == kWholeRow) {
                store_y(D.row);
            } else {
                // an item of a split row: its fp32 partial out; the last of the row's items to
                // finish adds all of them up in item order and stores y_r
                float2* pp = reinterpret_cast<float2*>(a.part + static_cast<size_t>(D.part) * a.d) + 4 * g + t;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    __stcg(pp + 64 * c, make_float2(yacc[c][0], yacc[c][1]));
                    __stcg(pp + 64 * c + 32, make_float2(yacc[c][2], yacc[c][3]));
                    yacc[c][0] = yacc[c][1] = yacc[c][2] = yacc[c][3] = 0.0f;
                }
                __threadfence();
                __syncwarp();
                int h = -1, nseg = 0;
                if (lane == 0) {
                    const int hh = __ldcg(&a.items[D.part].h);
                    const int ns = __ldcg(&a.heavy[hh].nseg);
                    if (atomicAdd(&a.heavy[hh].done, 1) == ns - 1) {
                        h = hh;
                        nseg = ns;
                    }
                }
                h = __shfl_sync(0xffffffffu, h, 0);
                nseg = __shfl_sync(0xffffffffu, nseg, 0);
                if (h >= 0) {
                    __threadfence();
                    for (int sg = 0; sg < nseg; ++sg) {
                        const float2* ps =
                            reinterpret_cast<const float2*>(a.part + static_cast<size_t>(h + sg) * a.d) + 4 * g + t;
#pragma unroll
                        for (int c = 0; c < NC; ++c) {
                            const float2 v0 = __ldcg(ps + 64 * c), v1 = __ldcg(ps + 64 * c + 32);
                            yacc[c][0] += v0.x;
                            yacc[c][1] += v0.y;
                            yacc[c][2] += v1.x;
                            yacc[c][3] += v1.y;
                        }
                    }
                    store_y(D.row);
                }
            }
        }
        __syncwarp();  // every lane is done with slot s before it is refilled
        ++n_done;
        issue();
        __syncwarp();  // the new slot's descriptor is visible to every lane
    }
    // After a timed-out wait: let the copies still in flight land before the CTA exits.
    for (int i = n_done; i < n_issued; ++i)
        wait_bounded(&bar[i % S], static_cast<uint32_t>(i / S) & 1u, nullptr, a.status, a.wait_ns);
}

// ------------------------------------------------------------------------------------------
// Work plan of the bulk kernel: one thread per token row, warps of 32 consecutive rows. A row's
// nonzeros are counted as the walk counts them (a tile count above T counts as 0), with eight
// loads in flight per thread (the counts are L2-resident). Rows with more than seg nonzeros
// get ceil(nnz / seg) consecutive items while the item list has room (one atomic per warp
// reserves the warp's items); the other rows go to the list of their class (above kClassA
// nonzeros, above kClassB, the rest). hdr[1..4] (zero at launch): items reserved, rows per class.
// The walk's work counter and the plan's counts set to zero, as a programmatic dependent of the
// kernel before it on the stream (normally the gate GEMM): it waits for that grid, then lets the plan
// kernel be scheduled. One warp.
__global__ void __launch_bounds__(32) zero_header_kernel(int* __restrict__ hdr, int n)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x < n) hdr[threadIdx.x] = 0;
}

__global__ void __launch_bounds__(128) split_plan_kernel(const uint16_t* __restrict__ cnt, int N, int nt, int T,
                                                         int seg, int item_cap, int* __restrict__ hdr,
                                                         int* __restrict__ list,
                                                         SplitItem* __restrict__ items, HeavyRow* __restrict__ heavy)
{
    // the walk (launched as this grid's programmatic dependent) may be scheduled now; it waits for
    // this grid to complete before it reads the plan. This grid itself is the dependent of the
    // header-zeroing kernel: the counts it reads and the counters it adds to are ready after the wait.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r - lane >= N) return;  // whole warp past the end
    const bool live = r < N;
    int nnz = 0;
    if (live) {
        const uint16_t* cr = cnt + static_cast<size_t>(r) * nt;
        int t = 0;
        for (; t + 8 <= nt; t += 8) {
            int c[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) c[k] = __ldg(cr + t + k);
#pragma unroll
            for (int k = 0; k < 8; ++k) nnz += c[k] > T ? 0 : c[k];
        }
        for (; t < nt; ++t) {
            const int c = __ldg(cr + t);
            nnz += c > T ? 0 : c;
        }
    }
    const bool want = live && nnz > seg;
    const int nseg = want ? (nnz + seg - 1) / seg : 0;
    int inc = nseg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
    }
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    int base0 = 0;
    if (lane == 0 && tot > 0) base0 = atomicAdd(&hdr[1], tot);
    const int base = __shfl_sync(0xffffffffu, base0, 0) + inc - nseg;
    bool split = false;
    if (want) {
        if (static_cast<long long>(base) + nseg <= item_cap) {
            split = true;
            heavy[base] = HeavyRow{r, nseg, base, 0};
            for (int sg = 0; sg < nseg; ++sg)
                items[base + sg] = SplitItem{r, static_cast<int>(static_cast<long long>(sg) * nnz / nseg),
                                             static_cast<int>(static_cast<long long>(sg + 1) * nnz / nseg), base};
        } else {  // no room: the reserved items that fall inside the list are left empty
            for (int sg = 0; sg < nseg && base + sg < item_cap; ++sg) items[base + sg] = SplitItem{0, 0, 0, kSkipPart};
        }
    }
    const int cls = (!live || split) ? -1 : (nnz > kClassA ? 0 : (nnz > kClassB ? 1 : 2));
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const unsigned m = __ballot_sync(0xffffffffu, cls == k);
        int b = 0;
        if (lane == 0 && m) b = atomicAdd(&hdr[2 + k], __popc(m));
        b = __shfl_sync(0xffffffffu, b, 0);
        if (cls == k) list[static_cast<size_t>(k) * N + b + __popc(m & below)] = r;
    }
}

// ------------------------------------------------------------------------------------------
// Launch

template <typename E, typename K>
static twell_status launch_persistent(K kern, const RowArgs<E>& a, size_t smem, int groups_per_cta, cudaStream_t s)
{
    twell_host::DevInfo di;
    if (twell_host::dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    if (smem > di.max_smem_optin) return TWELL_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return TWELL_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kCtaThreads, smem) != cudaSuccess || per_sm < 1)
        return TWELL_ERR_CUDA;
    if (cudaMemsetAsync(a.tickets, 0, sizeof(int), s) != cudaSuccess) return TWELL_ERR_CUDA;
    const int need = (a.N + groups_per_cta - 1) / groups_per_cta;  // CTAs until every group has a row
    int grid = di.sm_count * per_sm;
    if (grid > need) grid = need;
    kern<<<grid, kCtaThreads, smem, s>>>(a);
    return twell_host::launch_status();
}

template <typename E, int CPL, int G>
static twell_status launch_rows(const RowArgs<E>& a, cudaStream_t s)
{
    return launch_persistent(ffn_rows_kernel<E, CPL, G>, a, RowSmem<CPL>::cta_bytes(a.nt), kCtaWarps / G, s);
}

template <int CPLX, int R>
static twell_status launch_mma(const RowArgs<__nv_bfloat16>& a, cudaStream_t s)
{
    return launch_persistent(ffn_mma_kernel<CPLX, R>, a, MmaSmem<CPLX>::cta_bytes(a.nt), kCtaWarps, s);
}

template <int NS, int S, int WPC, bool F16DOWN>
static twell_status launch_bulk_k(const RowArgs<__nv_bfloat16>& a, cudaStream_t s)
{
    auto kern = ffn_bulk_kernel<NS, S, WPC, F16DOWN>;
    const size_t smem = static_cast<size_t>(WPC) * BulkLayout<NS>::warp_bytes(S, a.nt);
    twell_host::DevInfo di;
    if (twell_host::dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    if (smem > di.max_smem_optin) return TWELL_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return TWELL_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * WPC, smem) != cudaSuccess || per_sm < 1)
        return TWELL_ERR_CUDA;
    // the work counter and the plan's counts start at zero (a dependent one-warp kernel rather than a
    // memset, so that the gate, this, the plan and the walk chain as programmatic dependents); the
    // plan splits the long rows
    cudaLaunchConfig_t zc = {};
    cudaLaunchAttribute zattr[1];
    zattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    zattr[0].val.programmaticStreamSerializationAllowed = 1;
    zc.gridDim = dim3(1);
    zc.blockDim = dim3(32);
    zc.stream = s;
    zc.attrs = zattr;
    zc.numAttrs = 1;
    if (cudaLaunchKernelEx(&zc, zero_header_kernel, a.tickets, 5) != cudaSuccess) return TWELL_ERR_CUDA;
    RowArgs<__nv_bfloat16> b = a;
    b.split = 1;
    // Items of up to 128 nonzeros; for a small batch the largest power of two with at least one item
    // per resident warp if rows carried 32 nonzeros (seg <= 32 N / warps), but no fewer than 4.
    int seg = kSplitSeg;
    const long long warps = static_cast<long long>(di.sm_count) * per_sm * WPC;
    while (seg > kSplitSegMin && seg * warps > 32ll * a.N) seg >>= 1;
    cudaLaunchConfig_t pc = zc;
    pc.gridDim = dim3((a.N + 127) / 128);
    pc.blockDim = dim3(128);
    if (cudaLaunchKernelEx(&pc, split_plan_kernel, a.cnt, a.N, a.nt, a.T, seg, a.item_cap, a.tickets,
                           const_cast<int*>(a.list), const_cast<SplitItem*>(a.items), a.heavy) != cudaSuccess)
        return TWELL_ERR_CUDA;
    if (twell_host::launch_status() != TWELL_OK) return TWELL_ERR_CUDA;
    // a warp per work item at most: the rows plus the items split rows can be cut into
    const long long most_items = static_cast<long long>(a.N) * ((a.f + seg - 1) / seg);
    const long long work = a.N + (most_items < a.item_cap ? most_items : a.item_cap);
    const long long need = (work + WPC - 1) / WPC;
    int grid = di.sm_count * per_sm;
    if (grid > need) grid = static_cast<int>(need);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * WPC);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, b) != cudaSuccess) return TWELL_ERR_CUDA;
    return twell_host::launch_status();
}

template <int NS, int S, int WPC>
static twell_status launch_bulk(const RowArgs<__nv_bfloat16>& a, cudaStream_t s)
{
    return a.f16down ? launch_bulk_k<NS, S, WPC, true>(a, s) : launch_bulk_k<NS, S, WPC, false>(a, s);
}

// Kernel and layout for d_model = nchunks 16-byte chunks: the tensor-core kernel where it applies,
// else chunks per lane (CPL) and warps per row (G) of the general kernel.
template <typename E>
static twell_status run_fused(const RowArgs<E>& a, cudaStream_t s)
{
    if constexpr (std::is_same<E, __nv_bfloat16>::value) {
        const bool a32 = (reinterpret_cast<uintptr_t>(a.Wu) % 32 == 0) && (reinterpret_cast<uintptr_t>(a.Wd) % 32 == 0);
        // one warp per row: a warp's registers hold at most 2048 columns of y_r. Wider rows go to
        // the general kernel (two warps per row), which measured faster at 2560 columns (1.43 ms)
        // than this kernel with two warps per row (1.51 ms) on the 2B-like layer
        // the bulk-copy kernel where its ring fits in shared memory (d_model 512 .. 3072); 8 warps
        // per SM with a two-slot ring measured fastest on the 2048-wide layer (0.189-0.209 ms; three
        // slots and 6 warps 0.233, four slots and 4 warps 0.311, two warps per row 0.234)
        if (a.d % 256 == 0 && a.d >= 512 && a.d <= 3072) {
            twell_status st = TWELL_ERR_UNSUPPORTED;
            switch (a.d / 256) {
            case 2: st = launch_bulk<2, 2, 8>(a, s); break;
            case 3: st = launch_bulk<3, 2, 8>(a, s); break;
            case 4: st = launch_bulk<4, 2, 8>(a, s); break;
            case 5: st = launch_bulk<5, 2, 8>(a, s); break;
            case 6: st = launch_bulk<6, 2, 8>(a, s); break;
            case 7: st = launch_bulk<7, 2, 8>(a, s); break;
            case 8: st = launch_bulk<8, 2, 8>(a, s); break;
            case 10: st = launch_bulk<10, 2, 7>(a, s); break;
            case 12: st = launch_bulk<12, 2, 6>(a, s); break;
            default: break;
            }
            if (st != TWELL_ERR_UNSUPPORTED || a.f16down) return st;  // else: ring too large for shared memory
        }
        if (a.f16down) return TWELL_ERR_UNSUPPORTED;  // the other kernels read Wd as bf16
        if (a32 && a.d % 256 == 0) {
            switch (a.d / 256) {
            case 2: return launch_mma<2, 4>(a, s);
            case 4: return launch_mma<4, 3>(a, s);
            case 5: return launch_mma<5, 3>(a, s);
            case 6: return launch_mma<6, 3>(a, s);
            case 8: return launch_mma<8, 3>(a, s);
            default: break;
            }
        }
    }
    const int n = a.nchunks;
    if (n <= 32 * 2) return launch_rows<E, 2, 1>(a, s);
    if (n <= 32 * 4) return launch_rows<E, 4, 1>(a, s);
    if (n <= 32 * 8) return launch_rows<E, 8, 1>(a, s);
    if (n <= 64 * 5) return launch_rows<E, 5, 2>(a, s);
    if (n <= 64 * 8) return launch_rows<E, 8, 2>(a, s);
    if (n <= 128 * 8) return launch_rows<E, 8, 4>(a, s);
    return TWELL_ERR_UNSUPPORTED;
}

}  // namespace twell

size_t twell_host::fused_ws_bytes(int N, int d, int f) { return twell::FusedWs(N, d, f).total; }

using namespace twell_host;

// The bulk kernel's share of the workspace (see FusedWs); the first word is every kernel's counter.
template <typename E>
static void set_split_ws(twell::RowArgs<E>& p, void* ws, int N, int d, int f)
{
    const twell::FusedWs L(N, d, f);
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.item_cap = L.item_cap;
    p.list = reinterpret_cast<const int*>(w + L.list);
    p.items = reinterpret_cast<const twell::SplitItem*>(w + L.items);
    p.heavy = reinterpret_cast<twell::HeavyRow*>(w + L.heavy);
    p.part = reinterpret_cast<float*>(w + L.part);
}

extern "C" twell_status twell_ffn_fused_fwd(const void* x, const void* Wu_s, const void* Wd_s, const twell_packed* a,
                                            int32_t N, int32_t d, int32_t f, twell_dtype dtype, void* y, void* ws,
                                            size_t ws_bytes, int32_t* dev_status, void* stream)
{
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
    if (ws == nullptr || ws_bytes < twell_workspace_bytes(TWELL_OP_FFN_FUSED_FWD, N, d, f, a->tile, 0, 0))
        return TWELL_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(Wu_s) || !aligned16(Wd_s) || !aligned16(y) || !aligned16(ws))
        return TWELL_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int vals_bf16 = a->dtype == TWELL_BF16 ? 1 : 0;
    if (dtype == TWELL_BF16) {
        using bf = __nv_bfloat16;
        twell::RowArgs<bf> p{static_cast<const bf*>(x), static_cast<const bf*>(Wu_s), static_cast<const bf*>(Wd_s),
                             a->vals, a->idx, a->cnt, static_cast<bf*>(y), static_cast<int*>(ws), dev_status,
                             N, d, f, a->tile, nt, d / twell::Elem<bf>::kPer16B, vals_bf16};
        p.wait_ns = twell_host::wait_limit_ns();
        set_split_ws(p, ws, N, d, f);
        return twell::run_fused(p, s);
    }
    twell::RowArgs<float> p{static_cast<const float*>(x), static_cast<const float*>(Wu_s),
                            static_cast<const float*>(Wd_s), a->vals, a->idx, a->cnt, static_cast<float*>(y),
                            static_cast<int*>(ws), dev_status, N, d, f, a->tile, nt, d / twell::Elem<float>::kPer16B, 0};
    p.wait_ns = twell_host::wait_limit_ns();
    return twell::run_fused(p, s);
}

extern "C" twell_status twell_ffn_fused_fwd_f16down(const void* x, const void* Wu_s, const void* Wd16_s,
                                                    const twell_packed* a, int32_t N, int32_t d, int32_t f, void* y,
                                                    void* ws, size_t ws_bytes, int32_t* dev_status, void* stream)
{
    if (Wu_s == nullptr || Wd16_s == nullptr || a == nullptr || dev_status == nullptr) return TWELL_ERR_INVALID;
    if ((x == nullptr || y == nullptr) && N != 0) return TWELL_ERR_INVALID;
    if (N < 0 || d <= 0 || f <= 0 || d % 8 != 0) return TWELL_ERR_INVALID;
    if (!dtype_ok(a->dtype)) return TWELL_ERR_UNSUPPORTED;
    if (d % 256 != 0 || d < 512 || d > 3072) return TWELL_ERR_UNSUPPORTED;
    twell_status st = check_packed(a, N, f, a->tile, a->dtype);
    if (st != TWELL_OK) return st;
    const int nt = (f + a->tile - 1) / a->tile;
    if (nt > twell::kMaxTiles) return TWELL_ERR_UNSUPPORTED;
    if (N == 0) return TWELL_OK;
    if (ws == nullptr || ws_bytes < twell_workspace_bytes(TWELL_OP_FFN_FUSED_FWD, N, d, f, a->tile, 0, 0))
        return TWELL_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(Wu_s) || !aligned16(Wd16_s) || !aligned16(y) || !aligned16(ws))
        return TWELL_ERR_INVALID;
    using bf = __nv_bfloat16;
    twell::RowArgs<bf> p{static_cast<const bf*>(x), static_cast<const bf*>(Wu_s), static_cast<const bf*>(Wd16_s),
                         a->vals, a->idx, a->cnt, static_cast<bf*>(y), static_cast<int*>(ws), dev_status,
                         N, d, f, a->tile, nt, d / twell::Elem<bf>::kPer16B, a->dtype == TWELL_BF16 ? 1 : 0};
    p.wait_ns = twell_host::wait_limit_ns();
    p.f16down = 1;
    set_split_ws(p, ws, N, d, f);
    return twell::run_fused(p, static_cast<cudaStream_t>(stream));
}

namespace {
// bf16 -> fp16, one element per thread in a grid-stride loop. A finite value that leaves the fp16
// range (|w| > 65504) is recorded as TWELL_ERR_DEVICE_CHECK; it is stored as the infinity it rounds to.
__global__ void convert_f16_kernel(const __nv_bfloat16* __restrict__ src, __half* __restrict__ dst, size_t n,
                                   int32_t* status)
{
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float v = __bfloat162float(src[i]);
        const __half h = __float2half_rn(v);
        if (isfinite(v) && __hisinf(h)) twell::report(status, TWELL_ERR_DEVICE_CHECK);
        dst[i] = h;
    }
}
// src [rows, cols] bf16 -> dst [cols, rows] fp16 through 32 x 32 shared-memory tiles (reads and writes
// coalesced); an overflow of the fp16 range is recorded as in convert_f16_kernel.
__global__ void __launch_bounds__(256) convert_f16_t_kernel(const __nv_bfloat16* __restrict__ src,
                                                            __half* __restrict__ dst, int rows, int cols,
                                                            int32_t* status)
{
    __shared__ float tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int j = threadIdx.y; j < 32; j += 8) {
        const int r = r0 + j, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[j][threadIdx.x] = __bfloat162float(src[static_cast<size_t>(r) * cols + c]);
    }
    __syncthreads();
    for (int j = threadIdx.y; j < 32; j += 8) {
        const int c = c0 + j, r = r0 + threadIdx.x;
        if (r < rows && c < cols) {
            const float v = tile[threadIdx.x][j];
            const __half h = __float2half_rn(v);
            if (isfinite(v) && __hisinf(h)) twell::report(status, TWELL_ERR_DEVICE_CHECK);
            dst[static_cast<size_t>(c) * rows + r] = h;
        }
    }
}
}  // namespace

extern "C" twell_status twell_convert_f16_transposed(const void* src, void* dst, int32_t rows, int32_t cols,
                                                     int32_t* dev_status, void* stream)
{
    if (rows < 0 || cols < 0 || dev_status == nullptr) return TWELL_ERR_INVALID;
    if (rows == 0 || cols == 0) return TWELL_OK;
    if (src == nullptr || dst == nullptr) return TWELL_ERR_INVALID;
    if ((rows + 31) / 32 > 65535) return TWELL_ERR_UNSUPPORTED;
    const dim3 grid((cols + 31) / 32, (rows + 31) / 32);
    convert_f16_t_kernel<<<grid, dim3(32, 8), 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(src), static_cast<__half*>(dst), rows, cols, dev_status);
    return twell_host::launch_status();
}

extern "C" twell_status twell_convert_f16(const void* src, void* dst, int64_t n, int32_t* dev_status, void* stream)
{
    if (n < 0 || dev_status == nullptr) return TWELL_ERR_INVALID;
    if (n == 0) return TWELL_OK;
    if (src == nullptr || dst == nullptr) return TWELL_ERR_INVALID;
    twell_host::DevInfo di;
    if (twell_host::dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    const long long blocks_needed = (n + 255) / 256;
    const int grid = static_cast<int>(blocks_needed < 8ll * di.sm_count ? blocks_needed : 8ll * di.sm_count);
    convert_f16_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(src), static_cast<__half*>(dst), static_cast<size_t>(n), dev_status);
    return twell_host::launch_status();
}
