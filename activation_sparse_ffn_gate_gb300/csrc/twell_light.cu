// twell_light.cu -- the light rows of the hybrid training format on the tensor cores.
//
// A light row r keeps n_r <= K gate activations (column j, value a) in the sparse block of the
// hybrid format ([TG] "Обучение"; [TC] §3). Per kept entry the forward pass needs the dot product
// u = x_r . Wu_s[j] and the update y_r += h Wd_s[j] (h = a u); the backward pass needs
// dh = dy_r . Wd_s[j] and the update dx_r += du Wu_s[j] + dg Wg_s[j]. Neither forms a product of
// two dense matrices ([TG] "Обучение"): both are walks over the kept entries, organised like the
// inference walk of twell_ffn.cu.
//
// One warp per token row, rows taken from a counter. Lane 0 copies, per entry, the whole weight
// rows it needs (and the row vector x_r or dy_r at the row's first entry) into one slot of the
// warp's two-slot shared-memory ring with 1-D bulk copies (cp.async.bulk) completing on the slot's
// mbarrier, one entry ahead across row boundaries. Chunk c is columns [128c, 128c + 128) of
// d_model, with V[k][m] = v[128c + 8k + m] and W[k][n] = row[128c + 8k + n] (k < 16; m, n < 8):
//   dot:    mma.sync m16n8k16 with A = V^T (rows 0..7), B = W: D[m][m] summed over the chunks is
//           v . row; the eight diagonal lanes sum it in three xor steps and all hold the result;
//   update: A = s I (only the diagonal lanes hold s), B = W, so D += s W: the 16 x 8 accumulator of
//           chunk c holds out[128c + 8m + n] in fp32; s goes in as bf16 hi = bf16(s) and
//           lo = bf16(s - hi), so it is carried to ~16 significant bits.
// Every mbarrier wait is bounded; on expiry the warp records TWELL_ERR_TIMEOUT, lets its copies in
// flight land and stops.
#include "twell_light.cuh"
#include "twell_mma.cuh"

namespace twell {

namespace {

constexpr int kLFirst = 1, kLLast = 2;
constexpr int kLSeg = 32;  // entries of a row held in lane registers at a time

struct LightArgs {
    const __nv_bfloat16* v;   // x (forward) or dy (backward), [N, d]
    const __nv_bfloat16* W0;  // row of the dot product: Wu_s (forward), Wd_s (backward)
    const __nv_bfloat16* W1;  // first update row: Wd_s (forward), Wu_s (backward)
    const __nv_bfloat16* W2;  // second update row: Wg_s (backward)
    const float* ha;          // [N, K] a at the kept entries
    const uint16_t* hcol;     // [N, K] columns
    const uint16_t* hcnt;     // [N] entries per row, 0xFFFF for a backup row
    float* hu;                // [N, K] u: written by the forward, read by the backward
    __nv_bfloat16* y;         // forward output
    float* dx;                // backward output
    float* ent;               // backward: [N, K, 3] {h, du, dg}
    double* l1acc;            // forward: += sum |h|
    int* tickets;             // row counter, zero at launch
    int32_t* status;
    int N, d, f, K;
    float l1_scale;
    uint64_t wait_ns;
};

// Per warp: S slots of R bf16 rows of d_model (the weight rows of one entry, then the row vector
// at a row's first entry), S descriptors, S mbarriers.
template <int NS, int R>
struct LightLayout {
    static constexpr uint32_t kRow = 512u * NS;
    static constexpr uint32_t kSlot = R * kRow;
    __host__ __device__ static size_t warp_bytes(int S) { return (static_cast<size_t>(S) * (kSlot + 32 + 8) + 127) & ~size_t(127); }
};

struct __align__(16) LightDesc {
    int row, flags, e, pad;
    float a, u, pad0, pad1;
};

// The entries of the warp's rows in issue order. The row being issued holds one 32-entry segment
// in lane registers (lane k: entry base + k); the next row's count and first segment are loaded a
// row ahead, and the ticket of the row after that is taken a row before its loads.
template <bool BWD>
struct LightStream {
    int lane;
    int row, n, base, pos;  // row being issued (N: none left), its entry count, segment start, next entry
    int sj;
    float sa, su;
    int nrow, nn, nj;
    float na, nu;
    int tk;  // lane 0

    __device__ void load_segment(const LightArgs& a, int r, int b, int& j, float& av, float& uv) const
    {
        j = 0;
        av = uv = 0.0f;
        if (r < a.N && b + lane < a.K) {
            const size_t e = static_cast<size_t>(r) * a.K + b + lane;
            j = a.hcol[e];
            av = a.ha[e];
            if (BWD) uv = a.hu[e];
        }
    }
    __device__ void load_next(const LightArgs& a, int r)
    {
        nrow = r < a.N ? r : a.N;
        nn = r < a.N ? static_cast<int>(a.hcnt[r]) : 0;
        load_segment(a, r, 0, nj, na, nu);
        // the row vector of that row, copied into a slot a row from now, on its way from HBM to L2
        if (lane == 0 && r < a.N) bulk_prefetch_l2(a.v + static_cast<size_t>(r) * a.d, static_cast<uint32_t>(a.d) * 2u);
    }
    __device__ void take_ticket(const LightArgs& a)
    {
        tk = 0;
        if (lane == 0) tk = atomicAdd(a.tickets, 1);
    }
    __device__ void advance(const LightArgs& a)
    {
        row = nrow;
        n = nn;
        sj = nj;
        sa = na;
        su = nu;
        base = pos = 0;
        load_next(a, __shfl_sync(0xffffffffu, tk, 0));
        take_ticket(a);
    }
    __device__ void init(const LightArgs& a, int lane_)
    {
        lane = lane_;
        take_ticket(a);
        load_next(a, __shfl_sync(0xffffffffu, tk, 0));
        take_ticket(a);
        advance(a);
    }
    // Outputs of a light row that has no entries, and (forward) the padded u slots of any light row.
    __device__ void start_row(const LightArgs& a) const
    {
        if (!BWD)
            for (int k = n + lane; k < a.K; k += 32) a.hu[static_cast<size_t>(row) * a.K + k] = 0.0f;
        if (n != 0) return;
        if (BWD) {
            float4* o = reinterpret_cast<float4*>(a.dx + static_cast<size_t>(row) * a.d);
            for (int q = lane; q < a.d / 4; q += 32) o[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            uint4* o = reinterpret_cast<uint4*>(a.y + static_cast<size_t>(row) * a.d);
            for (int q = lane; q < a.d / 8; q += 32) o[q] = make_uint4(0, 0, 0, 0);
        }
    }
    // The next entry to issue, across row boundaries; false when the rows have run out.
    __device__ bool next(const LightArgs& a, LightDesc& D, int& j)
    {
        while (true) {
            if (row >= a.N) return false;
            if (n > a.K) {  // a backup row (0xFFFF), or a count past K (reported, skipped)
                if (n != 0xFFFF) report(a.status, TWELL_ERR_DEVICE_CHECK);
                advance(a);
                continue;
            }
            if (pos == 0) start_row(a);
            if (pos >= n) {
                advance(a);
                continue;
            }
            if (pos - base == kLSeg) {
                base += kLSeg;
                load_segment(a, row, base, sj, sa, su);
            }
            const int k = pos - base;
            j = __shfl_sync(0xffffffffu, sj, k);
            float av = __shfl_sync(0xffffffffu, sa, k);
            float uv = BWD ? __shfl_sync(0xffffffffu, su, k) : 0.0f;
            if (j >= a.f) {  // a column past d_ff: reported, contributes nothing
                report(a.status, TWELL_ERR_DEVICE_CHECK);
                j = 0;
                av = uv = 0.0f;
            }
            D.row = row;
            D.flags = (pos == 0 ? kLFirst : 0) | (pos == n - 1 ? kLLast : 0);
            D.e = row * a.K + pos;
            D.pad = 0;
            D.a = av;
            D.u = uv;
            D.pad0 = D.pad1 = 0.0f;
            ++pos;
            return true;
        }
    }
};

// Warp-level products over a bf16 row of d_model = 256 * NS held in shared memory (lane address
// base + 16 * lane: ldmatrix row addresses of a 512-byte span).
template <int NS>
struct RowOps {
    static constexpr int NC = 2 * NS;
    // The row vector as the A operands of the dot products, one register quad per chunk: a0 and
    // a2 are the chunk's V^T blocks, a1 and a3 (rows 8..15 of A, whose products are never read) the
    // neighbouring chunk's, so one ldmatrix gives a whole operand.
    __device__ static void load_vec(uint32_t (&vq)[NC][4], uint32_t sbase, int lane)
    {
        const int mi = lane >> 3, mr = lane & 7;
        const uint32_t off_e = 16u * mr + ((mi & 1) ? 256u : 0u) + ((mi & 2) ? 128u : 0u);
        const uint32_t off_o = 16u * mr + ((mi & 1) ? 0u : 256u) + ((mi & 2) ? 128u : 0u);
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            ldsm_x4_trans(vq[2 * q], sbase + 512u * q + off_e);
            ldsm_x4_trans(vq[2 * q + 1], sbase + 512u * q + off_o);
        }
    }
    // v . row (row at lane address sl); the diagonal lanes, lane 0 among them, return it.
    __device__ static float dot(const uint32_t (&vq)[NC][4], uint32_t sl, bool diag, int g)
    {
        float uc[4][4];
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            uint32_t w[4];
            ldsm_x4_trans(w, sl + 512u * q);
            const uint32_t(&e)[4] = vq[2 * q];
            const uint32_t(&o)[4] = vq[2 * q + 1];
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
        return u;
    }
    // acc += s * row (row at lane address sl), s as bf16 hi + lo on the diagonal lanes (hmask).
    __device__ static void axpy(float (&acc)[NC][4], float s, uint32_t hmask, uint32_t sl)
    {
        const uint32_t hi2 = bf16x2_rn(s, s);
        const float lo = s - __uint_as_float(hi2 << 16);
        const uint32_t hd = hi2 & hmask, ld = bf16x2_rn(lo, lo) & hmask;
#pragma unroll
        for (int q = 0; q < NS; ++q) {
            uint32_t w[4];
            ldsm_x4_trans(w, sl + 512u * q);
            mma_bf16(acc[2 * q], hd, 0u, 0u, hd, w[0], w[1]);
            mma_bf16(acc[2 * q + 1], hd, 0u, 0u, hd, w[2], w[3]);
            mma_bf16(acc[2 * q], ld, 0u, 0u, ld, w[0], w[1]);
            mma_bf16(acc[2 * q + 1], ld, 0u, 0u, ld, w[2], w[3]);
        }
    }
};

// The work-ticket counter is reset by a dependent one-thread kernel (not a memset), so that the
// reset and the walk can both be launched early behind the producing kernel.
__global__ void zero_ticket_kernel(int* tickets)
{
    pdl_begin();
    *tickets = 0;
}

// NS: 256-column spans of d_model; S: ring slots per warp; WPC: warps per CTA; BWD: backward.
template <int NS, int S, int WPC, bool BWD>
__global__ void __launch_bounds__(32 * WPC, 1) light_kernel(const LightArgs a)
{
    constexpr int R = BWD ? 4 : 3;  // weight rows per entry, then the row vector
    constexpr int NW = R - 1;
    using L = LightLayout<NS, R>;
    using Ops = RowOps<NS>;
    constexpr int NC = 2 * NS;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    uint8_t* wbase = smem + warp * L::warp_bytes(S);
    LightDesc* desc = reinterpret_cast<LightDesc*>(wbase + S * L::kSlot);
    uint64_t* bar = reinterpret_cast<uint64_t*>(desc + S);
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    __syncwarp();
    pdl_begin();  // the barriers above touch shared memory only

    const uint64_t pol_w = policy_evict_last(), pol_v = policy_evict_first();
    const __nv_bfloat16* Wr[3] = {a.W0, a.W1, a.W2};
    LightStream<BWD> ls;
    ls.init(a, lane);

    int n_issued = 0;
    bool ended = false;
    auto issue = [&]() {
        if (ended) return;
        LightDesc D;
        int j = 0;
        if (!ls.next(a, D, j)) {
            ended = true;
            return;
        }
        const int s = n_issued % S;
        if (lane == 0) {
            desc[s] = D;
            uint8_t* slot = wbase + s * L::kSlot;
            mbar_arrive_expect_tx(&bar[s], (D.flags & kLFirst) ? R * L::kRow : NW * L::kRow);
#pragma unroll
            for (int w = 0; w < NW; ++w)
                bulk_load(slot + w * L::kRow, Wr[w] + static_cast<size_t>(j) * a.d, L::kRow, &bar[s], pol_w);
            if (D.flags & kLFirst)
                bulk_load(slot + NW * L::kRow, a.v + static_cast<size_t>(D.row) * a.d, L::kRow, &bar[s], pol_v);
        }
        ++n_issued;
    };

    const bool diag = (g >> 1) == t;
    const uint32_t hmask = diag ? ((g & 1) ? 0xFFFF0000u : 0x0000FFFFu) : 0u;
    uint32_t vq[NC][4];
    float acc[NC][4];  // out_r: chunk c, columns 128c + 8g + 2t (+1) and 128c + 64 + 8g + 2t (+1)
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        vq[c][0] = vq[c][1] = vq[c][2] = vq[c][3] = 0u;
        acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;
    }
    float l1 = 0.0f;
    for (int i = 0; i < S; ++i) issue();
    __syncwarp();
    int n_done = 0;
    while (n_done < n_issued) {
        const int s = n_done % S;
        const bool ok =
            __all_sync(0xffffffffu, wait_bounded<false, 20000>(&bar[s], static_cast<uint32_t>(n_done / S) & 1u,
                                                              nullptr, a.status, a.wait_ns));
        if (!ok) break;
        const LightDesc D = desc[s];
        const uint32_t sb = smem_u32(wbase + s * L::kSlot);
        const uint32_t sl = sb + 16u * lane;
        if (D.flags & kLFirst) Ops::load_vec(vq, sb + NW * L::kRow, lane);
        const float p = Ops::dot(vq, sl, diag, g);
        if constexpr (!BWD) {
            const float h = D.a * p;  // p = u
            if (lane == 0) {
                a.hu[D.e] = p;
                l1 += fabsf(h);
            }
            Ops::axpy(acc, h, hmask, sl + L::kRow);
        } else {
            const float h = D.a * D.u;  // p = dh
            const float sg = h > 0.0f ? 1.0f : (h < 0.0f ? -1.0f : 0.0f);
            const float gg = p + a.l1_scale * sg;
            const float du = gg * D.a, dg = gg * D.u;  // a > 0 at every kept entry
            if (lane == 0) {
                float* en = a.ent + static_cast<size_t>(D.e) * 3;
                en[0] = h;
                en[1] = du;
                en[2] = dg;
            }
            Ops::axpy(acc, du, hmask, sl + L::kRow);
            Ops::axpy(acc, dg, hmask, sl + 2 * L::kRow);
        }
        if (D.flags & kLLast) {
            if constexpr (!BWD) {
                uint32_t* yr = reinterpret_cast<uint32_t*>(a.y + static_cast<size_t>(D.row) * a.d) + 4 * g + t;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    yr[64 * c] = bf16x2_rn(acc[c][0], acc[c][1]);
                    yr[64 * c + 32] = bf16x2_rn(acc[c][2], acc[c][3]);
                }
            } else {
                float2* o = reinterpret_cast<float2*>(a.dx + static_cast<size_t>(D.row) * a.d) + 4 * g + t;
#pragma unroll
                for (int c = 0; c < NC; ++c) {  // streaming stores: dx must not push the weight rows out of L2
                    st_stream8(o + 64 * c, acc[c][0], acc[c][1]);
                    st_stream8(o + 64 * c + 32, acc[c][2], acc[c][3]);
                }
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;
        }
        __syncwarp();  // every lane is done with slot s before it is refilled
        ++n_done;
        issue();
        __syncwarp();  // the new slot's descriptor is visible to every lane
    }
    // After a timed-out wait: let the copies still in flight land before the CTA exits.
    for (int i = n_done; i < n_issued; ++i)
        wait_bounded(&bar[i % S], static_cast<uint32_t>(i / S) & 1u, nullptr, a.status, a.wait_ns);
    if (!BWD && lane == 0 && l1 != 0.0f) atomicAdd(a.l1acc, static_cast<double>(l1));
}

template <int NS, int S, int WPC, bool BWD>
twell_status launch_light(const LightArgs& a, cudaStream_t s)
{
    auto kern = light_kernel<NS, S, WPC, BWD>;
    const size_t smem = static_cast<size_t>(WPC) * LightLayout<NS, BWD ? 4 : 3>::warp_bytes(S);
    twell_host::DevInfo di;
    if (twell_host::dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    if (smem > di.max_smem_optin) return TWELL_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return TWELL_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * WPC, smem) != cudaSuccess || per_sm < 1)
        return TWELL_ERR_CUDA;
    if (twell_host::launch_dep(zero_ticket_kernel, dim3(1), dim3(1), 0, s, a.tickets) != TWELL_OK) return TWELL_ERR_CUDA;
    const int need = (a.N + WPC - 1) / WPC;
    int grid = di.sm_count * per_sm;
    if (grid > need) grid = need;
    if (twell_host::launch_dep(kern, dim3(grid), dim3(32 * WPC), smem, s, a) != TWELL_OK) return TWELL_ERR_CUDA;
    return twell_host::launch_status();
}

// Warps per CTA: as many two-slot rings as fit in shared memory, at most eight.
template <bool BWD>
twell_status run_light(const LightArgs& a, cudaStream_t s)
{
    switch (a.d) {
    case 512: return launch_light<2, 2, 8, BWD>(a, s);
    case 1024: return launch_light<4, 2, 8, BWD>(a, s);
    case 2048: return launch_light<8, 2, BWD ? 7 : 8, BWD>(a, s);
    case 2560: return launch_light<10, 2, BWD ? 5 : 7, BWD>(a, s);
    default: return TWELL_ERR_UNSUPPORTED;
    }
}

bool light_shape_ok(int N, int d, int K, const void* const* ptrs, int n)
{
    if (d != 512 && d != 1024 && d != 2048 && d != 2560) return false;
    if (static_cast<long long>(N) * K >= (1ll << 31)) return false;
    for (int i = 0; i < n; ++i)
        if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0) return false;
    return true;
}

}  // namespace
}  // namespace twell

twell_status twell_host::light_fwd_bulk(const void* x, const void* Wu_s, const void* Wd_s, int N, int d, int f,
                                        int K, const float* ha, const uint16_t* hcol, const uint16_t* hcnt, float* hu,
                                        void* y, double* l1acc, int* tickets, int32_t* status, cudaStream_t s)
{
    const void* p[] = {x, Wu_s, Wd_s, y};
    if (!twell::light_shape_ok(N, d, K, p, 4)) return TWELL_ERR_UNSUPPORTED;
    if (N == 0) return TWELL_OK;
    using bf = __nv_bfloat16;
    twell::LightArgs a{static_cast<const bf*>(x), static_cast<const bf*>(Wu_s), static_cast<const bf*>(Wd_s), nullptr,
                       ha, hcol, hcnt, hu, static_cast<bf*>(y), nullptr, nullptr, l1acc, tickets, status,
                       N, d, f, K, 0.0f, wait_limit_ns()};
    return twell::run_light<false>(a, s);
}

twell_status twell_host::light_bwd_bulk(const void* dy, const void* Wg_s, const void* Wu_s, const void* Wd_s, int N,
                                        int d, int f, int K, const float* ha, const float* hu, const uint16_t* hcol,
                                        const uint16_t* hcnt, float l1_scale, float* ent, float* dx, int* tickets,
                                        int32_t* status, cudaStream_t s)
{
    const void* p[] = {dy, Wg_s, Wu_s, Wd_s, dx};
    if (!twell::light_shape_ok(N, d, K, p, 5)) return TWELL_ERR_UNSUPPORTED;
    if (N == 0) return TWELL_OK;
    using bf = __nv_bfloat16;
    twell::LightArgs a{static_cast<const bf*>(dy), static_cast<const bf*>(Wd_s), static_cast<const bf*>(Wu_s),
                       static_cast<const bf*>(Wg_s), ha, hcol, hcnt, const_cast<float*>(hu), nullptr, dx, ent,
                       nullptr, tickets, status, N, d, f, K, l1_scale, wait_limit_ns()};
    return twell::run_light<true>(a, s);
}
