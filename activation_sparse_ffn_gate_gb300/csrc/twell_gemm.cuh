// twell_gemm.cuh -- persistent warp-specialised tcgen05 GEMM for sm_103a with pluggable epilogues.
//
//   C[M, N] = A[M, K] * B[K, N]     bf16 (or, with F16, fp16) operands, fp32 accumulation in
//                                     tensor memory (TMEM)
//
// A is K-major ([M, K] row-major) or MN-major ([K, M] row-major); B is K-major ([N, K] row-major,
// i.e. the "rows of W" layout) or MN-major ([K, N] row-major). Tiles are 128 x BN x 64; TMA
// writes each operand stage into shared memory with the 128-byte swizzle; one thread issues the
// tcgen05.mma instructions into a double-buffered TMEM accumulator, so the epilogue of one tile
// overlaps the main loop of the next.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
// warps 2..5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31, i.e. one row each).
//
// M and K may be read from device memory (rows of a device-side list, e.g. the hybrid backup
// rows), so a launch sized for an upper bound does only the work that exists.
//
// Split K (k_splits > 1, StoreF32; one CTA or one CTA pair per tile): the k-blocks of each tile are cut into
// k_splits near-equal ranges, each a work unit of its own, and split s stores its partial sum at
// out + s * split_stride; the caller adds the partials in split order (a fixed order, so the
// result does not depend on scheduling). For products with few rows and a long K (the hybrid
// backup rows), where whole tiles would leave most SMs idle.
//
// PAIR (A and B K-major): CTAs run in clusters of two on an SM pair, and one tcgen05.mma of
// cta_group::2 computes a 256 x BN tile. CTA r holds rows [128r, 128r + 128) of the A tile and
// rows [r BN/2, (r + 1) BN/2) of the B tile, both at the same shared-memory offsets, and its
// TMEM receives rows [128r, 128r + 128) of D. Per SM this halves the B bytes that TMA writes and
// that the tensor core reads from shared memory (the 1-SM 128 x 256 tile needs 96 B/clk of
// each, above what one SM's shared memory serves at the full MMA rate).
//   * Both CTAs' TMA loads complete on the even CTA's full[s] (expect_tx of both halves, armed
//     by the even CTA's producer); only the even CTA's MMA thread issues MMAs and commits.
//   * Its commits free stage s on both CTAs' empty[s] and signal both CTAs' tfull[a]; the
//     epilogue warps of both CTAs release an accumulator on the even CTA's tempty[a] (count 8).
//   * A cluster barrier after TMEM allocation and before deallocation keeps each CTA's
//     barriers, shared memory and TMEM alive while the other may still signal or write them.
//
// Every mbarrier wait is bounded (twell::wait_bounded). On a timeout the CTA raises its abort
// flag, every role leaves its loop, the producer waits (bounded) for the TMA copies it issued,
// the MMA thread waits (bounded) for its last tcgen05 operations, and TMEM is freed before exit.
#pragma once

#include <cuda_fp16.h>

#include "twell_common.cuh"

namespace twell {

enum class Epi : int {
    PackTwell = 0,   // ReLU + TwELL pack of the gate accumulator (fp32 or bf16 values)
    StoreF32 = 1,    // out[m, n] = acc (fp32)
    StoreBF16 = 2,   // out[m, n] = bf16(acc)
    ScatterBF16 = 3, // out[rowmap[m], n] = bf16(acc)
    AccumF32 = 4,    // out[m, n] += acc (fp32)
    ScatterF32 = 5,  // out[rowmap[m], n] = acc (fp32)
    MulBF16 = 6,     // out[m, n] = bf16(acc * aux[m, n]), aux bf16
    MulHiLoBF16 = 7, // v = acc * aux[m, n]: out[m, n] = hi = bf16(v), out[m, n + lo_offset] = bf16(v - hi)
    MulMaskF16 = 8,  // out[m, n] = fp16(acc * aux[m, n]) where bit n of mask row m is set, else 0; aux
                     // fp16 (may be out itself: each element is read before it is written, by one thread)
    GateUpF16 = 9,   // PAIR only: the even CTA's B rows come from B (Wg_s), the odd CTA's from B2 (Wu_s),
                     // for the same BN / 2 units, so a tile holds g and u of 256 rows x BN / 2 units;
                     // the epilogue packs ReLU(g) into the TwELL as PackTwell does (T = 64 or 128) and
                     // stores out[m, n] = fp16(a * u) (a = the packed value) where g > 0, else 0
};

struct GemmArgs {
    int M, N, K;             // extents; M and K are upper bounds when M_dyn / K_dyn are given
    const int32_t* M_dyn;    // optional device scalar: M = min(M, *M_dyn)
    const int32_t* K_dyn;    // optional device scalar: K = min(K, *K_dyn)
    int kb_split;            // B source period in k-blocks: block kb reads map (kb / kb_split) & 1 at
                             // k-block kb % kb_split (one map: kb_split larger than every kb)
    int k_splits;            // split K into this many ranges (0 or 1: no split; StoreF32 only)
    int a_box_rows;          // rows of A a stage loads (0: the whole 128-row tile); fewer when M is small,
                             // the tile's other rows then hold stale data whose products are never stored
    int64_t split_stride;    // elements between the partial outputs of consecutive splits
    // StoreBF16 with PAIR, no split: the last tail_split tiles (the partial last wave) are cut into
    // two K halves, each a unit that stores an fp32 partial at tail_part (per tail tile and half a
    // [256 x BN] block, rows and columns relative to the tile); the caller adds the halves. A caller
    // asks with tail_split = -max: launch_gemm splits the last wave when it fills at most half the
    // clusters and has at most max tiles, and reports the count it chose (0: none).
    int tail_split;
    float* tail_part;
    void* out;               // epilogue output
    int64_t ldo;             // its leading dimension (elements)
    const int32_t* rowmap;   // ScatterBF16: destination row of each m
    const void* aux;         // MulBF16, MulHiLoBF16: bf16 factor matrix [M, ldaux]
    int64_t ldaux;
    int64_t lo_offset;       // MulHiLoBF16: columns between a value's hi and lo parts
    const uint32_t* mask;    // MulMaskF16: bit n of word mask[m * ldmask + n / 32] selects column n of row m
    int64_t ldmask;
    // PackTwell
    int vals_f32;  // packed values stored as fp32 (else bf16, rounded to nearest even)
    void* vals;
    uint8_t* idx;
    uint16_t* cnt;
    int T, nt;
    // launched as a programmatic dependent of the previous kernel on the stream: the prologue
    // (barriers, TMEM, tensor-map prefetch) overlaps that kernel's last wave, and every thread
    // waits for it to complete (griddepcontrol.wait) before any role starts; with M_dyn / K_dyn the
    // wait comes first, before the extents are read
    int pdl;
    // status
    int32_t* status;
    uint64_t wait_limit_ns;
};

constexpr int kGemmThreads = 192;
constexpr int kBM = 128;
constexpr int kBK = 64;

template <int BN, bool PAIR = false>
struct GemmCfg {
    static constexpr uint32_t A_BYTES = kBM * kBK * 2;
    static constexpr uint32_t B_BYTES = (PAIR ? BN / 2 : BN) * kBK * 2;  // this CTA's share of B
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    // one CTA: as many stages as fit in 192 KB (4 at BN = 256, 6 at 128, 8 at 64, 9 at 32)
    static constexpr int STAGES = PAIR ? 7 : (196608 / STAGE_BYTES < 10 ? static_cast<int>(196608 / STAGE_BYTES) : 10);
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/;
};

template <int BN, bool A_MN, bool B_MN, Epi EPI, bool PAIR, bool F16 = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const GemmArgs g)
{
    static_assert(!PAIR || (!A_MN && !B_MN && BN == 256), "the CTA-pair tile is 256 x 256 with K-major operands");
    static_assert(EPI != Epi::GateUpF16 || PAIR, "the gate + up tile takes its two B operands from a CTA pair");
    // N extent of one tile: BN columns of C, or BN / 2 units (their g and u) with GateUpF16
    constexpr int TN = EPI == Epi::GateUpF16 ? BN / 2 : BN;
    using C = GemmCfg<BN, PAIR>;
    constexpr int CG = PAIR ? 2 : 1;
    constexpr int STAGES = C::STAGES;
    constexpr uint32_t IDESC = F16 ? idesc_f16_f32(CG * kBM, BN, A_MN, B_MN) : idesc_bf16_f32(CG * kBM, BN, A_MN, B_MN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * C::B_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // an extent read from the device is written by an earlier kernel: wait for it first
    if (g.pdl && (g.M_dyn != nullptr || g.K_dyn != nullptr)) asm volatile("griddepcontrol.wait;" ::: "memory");
    int M = g.M;
    if (g.M_dyn != nullptr) M = min(M, *g.M_dyn);
    int K = g.K;
    if (g.K_dyn != nullptr) K = min(K, *g.K_dyn);
    const int m_tiles = M > 0 ? (M + kBM - 1) / kBM : 0;
    const int n_tiles = (g.N + TN - 1) / TN;
    const int kbs = K > 0 ? (K + kBK - 1) / kBK : 0;
    // k-block ranges per tile: ks of them, each non-empty
    const int ks = (EPI != Epi::StoreF32 || g.k_splits <= 1) ? 1 : min(g.k_splits, max(kbs, 1));
    // work units: one 128 x BN tile per CTA, or with PAIR one 256 x BN tile per cluster, of which
    // this CTA holds the 128 rows of its rank (past M its loads read zeros and its epilogue
    // writes nothing)
    const int crank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    const bool leader = crank == 0;
    const int unit0 = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int ustride = PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
    const int tiles = (PAIR ? (m_tiles + 1) / 2 : m_tiles) * n_tiles;
    // tail split: the last ts tiles as two K halves each (units n_whole .. n_whole + 2 ts)
    const int ts = (EPI == Epi::StoreBF16 && PAIR && ks == 1 && kbs >= 2) ? min(max(g.tail_split, 0), tiles) : 0;
    const int n_whole = tiles - ts;
    const int units = kbs > 0 ? (ts > 0 ? n_whole + 2 * ts : tiles * ks) : 0;
    // unit u: tile u / ks, k-block range u % ks; past n_whole with a tail split: tile n_whole + (u - n_whole) / 2,
    // K half (u - n_whole) % 2
    auto tile_of = [&](int u) { return (ts == 0 || u < n_whole) ? u / ks : n_whole + ((u - n_whole) >> 1); };
    auto half_of = [&](int u) { return (ts == 0 || u < n_whole) ? -1 : ((u - n_whole) & 1); };
    auto tile_m0 = [&](int u) {
        const int tl = tile_of(u);
        return (PAIR ? 2 * (tl / n_tiles) + crank : tl / n_tiles) * kBM;
    };
    auto tile_n0 = [&](int u) { return (tile_of(u) % n_tiles) * TN; };
    auto kb_begin = [&](int u) {
        const int hh = half_of(u);
        if (hh >= 0) return hh ? kbs / 2 : 0;
        return static_cast<int>(static_cast<long long>(u % ks) * kbs / ks);
    };
    auto kb_end = [&](int u) {
        const int hh = half_of(u);
        if (hh >= 0) return hh ? kbs : kbs / 2;
        return static_cast<int>(static_cast<long long>(u % ks + 1) * kbs / ks);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4 * CG);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (EPI == Epi::GateUpF16 || g.kb_split < kbs) tma_prefetch_desc(&tmB2);
    }
    if (warp == 1) {
        tmem_alloc<CG>(tmem_slot, C::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // both CTAs' barriers and TMEM exist before either is used
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (g.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous grid's writes are visible
    // A kernel launched as this one's programmatic dependent may be scheduled now. It waits for this
    // grid to complete before it reads what this grid writes; only after this point, when every
    // kernel before this one has completed, so that it may read the weights before its own wait.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the even CTA's barriers, as shared::cluster addresses (PAIR)
    const uint32_t full_lead = PAIR ? mapa_shared(smem_u32(full), 0) : 0u;
    const uint32_t tempty_lead = PAIR ? mapa_shared(smem_u32(tempty), 0) : 0u;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int t = unit0; ok && t < units; t += ustride) {
                const int m0 = tile_m0(t);
                const int n0 = tile_n0(t);
                const int kb1 = kb_end(t);
                for (int kb = kb_begin(t); kb < kb1; ++kb) {
                    if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, g.status, g.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    uint8_t* a = sA + stage * C::A_BYTES;
                    uint8_t* b = sB + stage * C::B_BYTES;
                    const int k0 = kb * kBK;
                    if constexpr (PAIR) {
                        // this CTA's halves of A and B; both CTAs' copies complete on the even CTA's full[s]
                        if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                        const uint32_t fb = full_lead + stage * 8u;
                        tma_load_2d_pair(a, &tmA, k0, m0, fb);
                        if constexpr (EPI == Epi::GateUpF16)
                            tma_load_2d_pair(b, crank ? &tmB2 : &tmB, k0, n0, fb);
                        else
                            tma_load_2d_pair(b, &tmB, k0, n0 + crank * (BN / 2), fb);
                    } else {
                        mbar_arrive_expect_tx(&full[stage], g.a_box_rows > 0 && !A_MN
                                                                ? static_cast<uint32_t>(g.a_box_rows) * kBK * 2 + C::B_BYTES
                                                                : C::STAGE_BYTES);
                        if constexpr (!A_MN) {
                            tma_load_2d(a, &tmA, k0, m0, &full[stage]);
                        } else {
                            tma_load_2d(a, &tmA, m0, k0, &full[stage]);
                            tma_load_2d(a + 8192, &tmA, m0 + 64, k0, &full[stage]);
                        }
                        const CUtensorMap* tb = ((kb / g.kb_split) & 1) ? &tmB2 : &tmB;
                        const int kk = (kb % g.kb_split) * kBK;
                        if constexpr (!B_MN) {
                            tma_load_2d(b, tb, kk, n0, &full[stage]);
                        } else {
#pragma unroll
                            for (int s = 0; s < BN / 64; ++s)
                                tma_load_2d(b + s * 8192, tb, n0 + 64 * s, kk, &full[stage]);
                        }
                    }
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Wait (bounded, even after an abort) for every copy this thread issued to land, so
            // no TMA write into shared memory is still in flight when the CTA exits. With PAIR the
            // even CTA's full barriers count both CTAs' copies, and the cluster barrier at the end
            // holds the odd CTA until they have landed.
            if (leader)
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s))
                        wait_bounded(&full[s], (issued_phase >> s) & 1u, nullptr, g.status, g.wait_limit_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int t = unit0; ok && t < units; t += ustride) {
                if (!wait_bounded<PAIR>(&tempty[acc], acc_phase ^ 1u, abort_flag, g.status, g.wait_limit_ns)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                const int kb0 = kb_begin(t), kb1 = kb_end(t);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(&full[stage], phase, abort_flag, g.status, g.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + stage * C::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        // one MMA consumes K = 16: 32 bytes along a K-major row, 16 rows of an MN-major tile
                        const uint64_t da = A_MN ? desc_sw128(a_addr + k * 2048, 8192) : desc_sw128(a_addr + k * 32, 16);
                        const uint64_t db = B_MN ? desc_sw128(b_addr + k * 2048, 8192) : desc_sw128(b_addr + k * 32, 16);
                        tc_mma_f16<CG>(d_tmem, da, db, IDESC, (kb != kb0 || k != 0) ? 1u : 0u);
                    }
                    // frees this stage (in both CTAs with PAIR) once its MMAs have read it
                    if constexpr (PAIR) tc_commit_mc<CG>(&empty[stage], 0x3);
                    else tc_commit<CG>(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                // accumulator complete
                if constexpr (PAIR) tc_commit_mc<CG>(&tfull[acc], 0x3);
                else tc_commit<CG>(&tfull[acc]);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Wait (bounded) for every tcgen05 operation this thread issued before TMEM is freed.
            tc_commit<CG>(drain);
            wait_bounded(drain, 0, nullptr, g.status, g.wait_limit_ns);
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint32_t acc = 0, acc_phase = 0;
        for (int t = unit0; t < units; t += ustride) {
            int ok = 1;
            if (lane == 0) ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, g.status, g.wait_limit_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const int m0 = tile_m0(t);
            const int n0 = tile_n0(t);
            const int row = m0 + 32 * q + lane;
            const bool row_ok = row < M;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * BN;

            if constexpr (EPI == Epi::GateUpF16) {
                // columns [0, TN) of the accumulator hold g of units n0 .. n0 + TN, columns [TN, 2 TN)
                // u of the same units. Per T-wide column tile: ReLU + TwELL pack of g as below, and
                // h = a * u (a = the value as packed) stored as fp16 for every unit below ldo.
                const int T = g.T;
                __nv_bfloat16* vals16 = static_cast<__nv_bfloat16*>(g.vals);
                float* vals32 = static_cast<float*>(g.vals);
                __half* H = static_cast<__half*>(g.out);
                bool over = false;
                for (int tt = 0; tt < TN / T; ++tt) {
                    const int tile = n0 / T + tt;
                    const bool valid = row_ok && tile < g.nt;
                    const size_t slot = (static_cast<size_t>(row) * g.nt + tile) * static_cast<size_t>(T);
                    int c = 0;
                    for (int ch = 0; ch < T / 32; ++ch) {
                        float gv[32], uv[32];
                        tmem_ld_32x32b_x32(taddr + tt * T + ch * 32, gv);
                        tmem_ld_32x32b_x32(taddr + TN + tt * T + ch * 32, uv);
                        const int col0 = n0 + tt * T + ch * 32;
                        if (valid) {
#pragma unroll
                            for (int k = 0; k < 32; ++k) {
                                if (gv[k] > 0.0f) {
                                    if (g.vals_f32) {
                                        vals32[slot + c] = gv[k];
                                    } else {
                                        const __nv_bfloat16 b = __float2bfloat16_rn(gv[k]);
                                        vals16[slot + c] = b;
                                        gv[k] = __bfloat162float(b);
                                    }
                                    g.idx[slot + c] = static_cast<uint8_t>(ch * 32 + k);
                                    ++c;
                                }
                            }
                        }
                        if (row_ok && col0 < g.ldo) {  // ldo is a multiple of 32: whole chunks
                            uint4* o = reinterpret_cast<uint4*>(H + static_cast<size_t>(row) * g.ldo + col0);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uint32_t ow[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int k = 8 * i + 2 * e;
                                    const float h0 = gv[k] > 0.0f ? gv[k] * uv[k] : 0.0f;
                                    const float h1 = gv[k + 1] > 0.0f ? gv[k + 1] * uv[k + 1] : 0.0f;
                                    over |= !(fabsf(h0) < 65520.0f) || !(fabsf(h1) < 65520.0f);
                                    const __half2 hh = __floats2half2_rn(h0, h1);
                                    ow[e] = *reinterpret_cast<const uint32_t*>(&hh);
                                }
                                o[i] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                            }
                        }
                    }
                    if (valid) g.cnt[static_cast<size_t>(row) * g.nt + tile] = static_cast<uint16_t>(c);
                }
                if (over) report(g.status, TWELL_ERR_DEVICE_CHECK);
            } else if constexpr (EPI == Epi::PackTwell) {
                // ReLU + TwELL: per (row, T-wide column tile) keep g > 0 in ascending column order.
                const int T = g.T;
                __nv_bfloat16* vals16 = static_cast<__nv_bfloat16*>(g.vals);
                float* vals32 = static_cast<float*>(g.vals);
                for (int tt = 0; tt < BN / T; ++tt) {
                    const int tile = n0 / T + tt;
                    const bool valid = row_ok && tile < g.nt;
                    const size_t slot = (static_cast<size_t>(row) * g.nt + tile) * static_cast<size_t>(T);
                    int c = 0;
                    for (int ch = 0; ch < T / 32; ++ch) {
                        float v[32];
                        tmem_ld_32x32b_x32(taddr + tt * T + ch * 32, v);
                        if (valid) {
#pragma unroll
                            for (int k = 0; k < 32; ++k) {
                                if (v[k] > 0.0f) {
                                    if (g.vals_f32) vals32[slot + c] = v[k];
                                    else vals16[slot + c] = __float2bfloat16_rn(v[k]);
                                    g.idx[slot + c] = static_cast<uint8_t>(ch * 32 + k);
                                    ++c;
                                }
                            }
                        }
                    }
                    if (valid) g.cnt[static_cast<size_t>(row) * g.nt + tile] = static_cast<uint16_t>(c);
                }
            } else {
                const int thalf = half_of(t);
                for (int ch = 0; ch < BN / 32; ++ch) {
                    float v[32];
                    tmem_ld_32x32b_x32(taddr + ch * 32, v);
                    const int col0 = n0 + ch * 32;
                    if (!row_ok || col0 >= g.N) continue;
                    const int nvalid = min(32, g.N - col0);
                    if (EPI == Epi::StoreBF16 && thalf >= 0) {
                        // a K half of a tail tile: fp32 partial, rows and columns relative to the tile
                        const int lr = 32 * q + lane + (PAIR ? crank * kBM : 0);
                        float* o = g.tail_part +
                                   ((static_cast<size_t>(tile_of(t) - n_whole) * 2 + thalf) * (CG * kBM) + lr) * BN + ch * 32;
#pragma unroll
                        for (int k = 0; k < 32; k += 4)
                            if (k < nvalid) *reinterpret_cast<float4*>(o + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
                        continue;
                    }
                    if constexpr (EPI == Epi::StoreF32 || EPI == Epi::AccumF32 || EPI == Epi::ScatterF32) {
                        const int orow = (EPI == Epi::ScatterF32) ? g.rowmap[row] : row;
                        float* o = static_cast<float*>(g.out) + static_cast<size_t>(orow) * g.ldo + col0 +
                                   (ks > 1 ? static_cast<size_t>(t % ks) * g.split_stride : size_t(0));
                        if (nvalid == 32) {
#pragma unroll
                            for (int k = 0; k < 32; k += 4) {
                                float4 w = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
                                if constexpr (EPI == Epi::AccumF32) {
                                    const float4 p = *reinterpret_cast<const float4*>(o + k);
                                    w.x += p.x;
                                    w.y += p.y;
                                    w.z += p.z;
                                    w.w += p.w;
                                }
                                *reinterpret_cast<float4*>(o + k) = w;
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 32; ++k) {
                                if (k < nvalid) {
                                    if constexpr (EPI == Epi::AccumF32) o[k] += v[k];
                                    else o[k] = v[k];
                                }
                            }
                        }
                    } else if constexpr (EPI == Epi::MulMaskF16) {
                        const uint32_t km = g.mask[static_cast<size_t>(row) * g.ldmask + col0 / 32];
                        const uint4* ax = reinterpret_cast<const uint4*>(static_cast<const __half*>(g.aux) +
                                                                         static_cast<size_t>(row) * g.ldaux + col0);
                        uint4* o = reinterpret_cast<uint4*>(static_cast<__half*>(g.out) + static_cast<size_t>(row) * g.ldo +
                                                            col0);
                        uint4 av[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) av[i] = ax[i];  // col0 + 32 <= N: the columns are whole chunks
                        bool over = false;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t aw[4] = {av[i].x, av[i].y, av[i].z, av[i].w};
                            uint32_t ow[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c = 8 * i + 2 * e;
                                const float2 af = __half22float2(*reinterpret_cast<const __half2*>(&aw[e]));
                                const float h0 = ((km >> c) & 1u) ? af.x * v[c] : 0.0f;
                                const float h1 = ((km >> (c + 1)) & 1u) ? af.y * v[c + 1] : 0.0f;
                                over |= !(fabsf(h0) < 65520.0f) || !(fabsf(h1) < 65520.0f);
                                const __half2 hh = __floats2half2_rn(h0, h1);
                                ow[e] = *reinterpret_cast<const uint32_t*>(&hh);
                            }
                            o[i] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                        }
                        if (over) report(g.status, TWELL_ERR_DEVICE_CHECK);
                    } else {
                        const int orow = (EPI == Epi::ScatterBF16) ? g.rowmap[row] : row;
                        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(g.out) + static_cast<size_t>(orow) * g.ldo + col0;
                        if constexpr (EPI == Epi::MulBF16 || EPI == Epi::MulHiLoBF16) {  // v *= aux[row, col0 ..]
                            const __nv_bfloat16* ax = static_cast<const __nv_bfloat16*>(g.aux) +
                                                      static_cast<size_t>(row) * g.ldaux + col0;
                            if (nvalid == 32) {
#pragma unroll
                                for (int k = 0; k < 32; k += 8) {
                                    float f8[8];
                                    unpack16(*reinterpret_cast<const uint4*>(ax + k), f8,
                                             static_cast<__nv_bfloat16*>(nullptr));
#pragma unroll
                                    for (int e = 0; e < 8; ++e) v[k + e] *= f8[e];
                                }
                            } else {
#pragma unroll
                                for (int k = 0; k < 32; ++k)
                                    if (k < nvalid) v[k] *= __bfloat162float(ax[k]);
                            }
                        }
                        if constexpr (EPI == Epi::MulHiLoBF16) {  // hi, and the rounding remainder as lo
                            if (nvalid == 32) {
#pragma unroll
                                for (int k = 0; k < 32; k += 8) {
                                    float hi8[8], lo8[8];
#pragma unroll
                                    for (int e = 0; e < 8; ++e) {
                                        hi8[e] = __bfloat162float(__float2bfloat16_rn(v[k + e]));
                                        lo8[e] = v[k + e] - hi8[e];
                                    }
                                    *reinterpret_cast<uint4*>(o + k) = pack16(hi8, static_cast<__nv_bfloat16*>(nullptr));
                                    *reinterpret_cast<uint4*>(o + g.lo_offset + k) =
                                        pack16(lo8, static_cast<__nv_bfloat16*>(nullptr));
                                }
                            } else {
#pragma unroll
                                for (int k = 0; k < 32; ++k)
                                    if (k < nvalid) {
                                        const __nv_bfloat16 hb = __float2bfloat16_rn(v[k]);
                                        o[k] = hb;
                                        o[g.lo_offset + k] = __float2bfloat16_rn(v[k] - __bfloat162float(hb));
                                    }
                            }
                        } else if (nvalid == 32) {
#pragma unroll
                            for (int k = 0; k < 32; k += 8) {
                                float f8[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) f8[e] = v[k + e];
                                *reinterpret_cast<uint4*>(o + k) = pack16(f8, static_cast<__nv_bfloat16*>(nullptr));
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                if (k < nvalid) o[k] = __float2bfloat16_rn(v[k]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(tempty_lead + acc * 8u);
                else mbar_arrive(&tempty[acc]);
            }
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the pair's last copies, MMAs and arrivals have landed
    tc_fence_after();
    if (warp == 1) tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
}

}  // namespace twell

namespace twell_host {

// Operand description for the host launcher.
struct GemmOperand {
    const void* ptr;  // row-major matrix of 16-bit elements (bf16, or fp16 with F16)
    int64_t rows, cols, ld;
};

// Launch C = A * B with the tcgen05 kernel. A: [M, K] (a_mn = false) or [K, M] (a_mn = true);
// B: [N, K] (b_mn = false) or [K, N] (b_mn = true); B2 (optional) continues B along K from
// k-block kb_split on. Returns TWELL_ERR_CUDA on a tensor-map or launch failure.
template <int BN, bool A_MN, bool B_MN, twell::Epi EPI, bool PAIR = false, bool F16 = false>
twell_status launch_gemm(const GemmOperand& A, const GemmOperand& B, const GemmOperand* B2, twell::GemmArgs g,
                         cudaStream_t stream, int* tail_chosen = nullptr);

}  // namespace twell_host

namespace twell_host {

template <int BN, bool A_MN, bool B_MN, twell::Epi EPI, bool PAIR, bool F16>
twell_status launch_gemm(const GemmOperand& A, const GemmOperand& B, const GemmOperand* B2, twell::GemmArgs g,
                         cudaStream_t stream, int* tail_chosen)
{
    if (tail_chosen != nullptr) *tail_chosen = 0;
    static_assert(!PAIR || (!A_MN && !B_MN), "the CTA-pair GEMM takes K-major operands");
    using Cfg = twell::GemmCfg<BN, PAIR>;
    constexpr bool DUAL = EPI == twell::Epi::GateUpF16;
    constexpr int TN = DUAL ? BN / 2 : BN;
    if (PAIR && (B2 != nullptr) != DUAL) return TWELL_ERR_UNSUPPORTED;
    DevInfo di;
    if (dev_info(&di) != TWELL_OK) return TWELL_ERR_CUDA;
    if (di.max_smem_optin < Cfg::SMEM_BYTES) return TWELL_ERR_UNSUPPORTED;
    if (g.M <= 0 || g.N <= 0 || g.K <= 0) return TWELL_OK;
    CUtensorMap ta, tb, tb2;
    twell_status st;
    // A: K-major box = 64 (K) x 128 (M), or x M rounded up to 8 when M is below 128 (one tile, most
    // of whose rows would be zero fill); MN-major box = 64 (M) x 64 (K), two per stage.
    g.a_box_rows = (!PAIR && !A_MN && g.M_dyn == nullptr && g.M <= twell::kBM - 8) ? (g.M + 7) / 8 * 8 : 0;
    st = A_MN ? make_tmap_bf16(&ta, A.ptr, A.cols, A.rows, A.ld, 64, 64)
              : make_tmap_bf16(&ta, A.ptr, A.cols, A.rows, A.ld, 64, g.a_box_rows > 0 ? g.a_box_rows : twell::kBM);
    if (st != TWELL_OK) return st;
    // B: K-major box = 64 (K) x BN (N), or BN/2 rows per CTA with PAIR; MN-major box = 64 (N) x
    // 64 (K), BN/64 per stage.
    st = B_MN ? make_tmap_bf16(&tb, B.ptr, B.cols, B.rows, B.ld, 64, 64)
              : make_tmap_bf16(&tb, B.ptr, B.cols, B.rows, B.ld, 64, PAIR ? BN / 2 : BN);
    if (st != TWELL_OK) return st;
    if (B2 != nullptr) {
        st = B_MN ? make_tmap_bf16(&tb2, B2->ptr, B2->cols, B2->rows, B2->ld, 64, 64)
                  : make_tmap_bf16(&tb2, B2->ptr, B2->cols, B2->rows, B2->ld, 64, PAIR ? BN / 2 : BN);
        if (st != TWELL_OK) return st;
        if (DUAL) g.kb_split = 1 << 30;
    } else {
        tb2 = tb;
        g.kb_split = 1 << 30;
    }
    auto kern = twell::tc_gemm_kernel<BN, A_MN, B_MN, EPI, PAIR, F16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::SMEM_BYTES)) !=
        cudaSuccess)
        return TWELL_ERR_CUDA;
    g.wait_limit_ns = wait_limit_ns();
    const long long m_tiles = (g.M + twell::kBM - 1) / twell::kBM, n_tiles = (g.N + TN - 1) / TN;
    if (g.k_splits > 1 && EPI != twell::Epi::StoreF32) return TWELL_ERR_UNSUPPORTED;
    if constexpr (!PAIR) {
        const long long tiles = m_tiles * n_tiles * (g.k_splits > 1 ? g.k_splits : 1);
        const int grid = static_cast<int>(tiles < di.sm_count ? tiles : di.sm_count);
        if (!g.pdl) {
            kern<<<grid, twell::kGemmThreads, Cfg::SMEM_BYTES, stream>>>(ta, tb, tb2, g);
            return launch_status();
        }
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(twell::kGemmThreads);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2, g) != cudaSuccess) return TWELL_ERR_CUDA;
        return launch_status();
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.blockDim = dim3(twell::kGemmThreads);
        cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2 * static_cast<unsigned>(di.sm_count / 2));
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) return TWELL_ERR_CUDA;
        long long units = ((m_tiles + 1) / 2) * n_tiles * (g.k_splits > 1 ? g.k_splits : 1);
        if (g.tail_split < 0) {
            // split the last, partial wave of tiles into K halves when it fills at most half the pairs
            const long long tail = units % clusters;
            const int kbs = (g.K + twell::kBK - 1) / twell::kBK;
            g.tail_split = (EPI == twell::Epi::StoreBF16 && g.k_splits <= 1 && g.tail_part != nullptr && kbs >= 2 &&
                            units > clusters && tail > 0 && 2 * tail <= clusters && tail <= -g.tail_split)
                               ? static_cast<int>(tail)
                               : 0;
            units += g.tail_split;
            if (tail_chosen != nullptr) *tail_chosen = g.tail_split;
        }
        if (clusters > units) clusters = static_cast<int>(units);
        cfg.gridDim = dim3(2 * static_cast<unsigned>(clusters));
        cfg.numAttrs = g.pdl ? 2 : 1;
        if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2, g) != cudaSuccess) return TWELL_ERR_CUDA;
        return launch_status();
    }
}

}  // namespace twell_host
