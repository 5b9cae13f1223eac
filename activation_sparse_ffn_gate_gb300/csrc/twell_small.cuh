// twell_small.cuh -- the gate + TwELL pack of a batch of at most 16 tokens (decoding), as device
// phases shared by gate_small_kernel (twell_gate.cu) and the fused decode kernel (twell_decode.cu).
//
// The gate GEMM of a few tokens is a skinny one: Wg_s (d_ff x d_model, 23 MB on the 1.5B-like
// layer) is read once. A cluster of two CTAs owns one T-wide column tile, each CTA T/2 hidden units,
// so 2 * d_ff / T SMs share the read, and every CTA keeps 128 KB of weight loads in flight:
//   * 16 warps; warp w takes the 16-unit block w % (U/16) and every (16/(U/16))-th 64-element
//     span of d_model; per span each lane loads 32 contiguous bytes of its two units' rows
//     (16-byte read-only loads that skip L1) -- the k order inside a span is permuted the same way
//     for both operands, so the fragments come straight from those loads;
//   * the part of each row past a warp's first batch of spans is prefetched to L2 at the start, so
//     the later batches' loads hit L2;
//   * x (padded to 8 or 16 token rows, rows >= N zero) is staged in shared memory once, by
//     asynchronous copies in flight together with the first weight loads;
//   * products on mma.sync m16n8k16 (units as the 16 rows, tokens as the 8 columns), fp32
//     accumulation; the warps' partial sums over d_model are added in a fixed order, so g does not
//     depend on scheduling;
//   * the two CTAs of the cluster exchange nothing but their g values: after a cluster barrier,
//     CTA c packs tokens c, c + 2, ... over the whole tile, reading the other half from the peer's
//     shared memory (distributed shared memory), in ascending column order, as the tile epilogue
//     of the large-batch GEMM does ([AIM] ¶3; [PUL] ¶3; [TC] §2).
// An entry is kept iff its fp32 g is > 0, and its value stored as g (fp32) or bf16(g).
#pragma once

#include <cooperative_groups.h>

#include "twell_common.cuh"
#include "twell_mma.cuh"

namespace twell {

constexpr int kSmallWarps = 16;
constexpr int kSmallMaxN = 16;

// 16-byte asynchronous copy global -> shared; src_bytes 0 fills the 16 bytes with zeros (nothing is read).
__device__ __forceinline__ void small_cp_async16(void* smem_dst, const void* gsrc, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(src_bytes)
                 : "memory");
}

// Shared memory of one CTA (byte offsets): staged x, the warps' partial g, g of the CTA's units.
struct SmallGateLayout {
    size_t x_stride, x, part, g, total;
    __host__ __device__ SmallGateLayout(int NB, int T, int d)
    {
        const int U = T / 2, KS = kSmallWarps / (U / 16);
        x_stride = static_cast<size_t>(d) * 2 + 16;  // 16-byte pad: the 8 token rows fall in different banks
        x = 0;
        part = static_cast<size_t>(8 * NB) * x_stride;
        g = part + static_cast<size_t>(KS) * U * 8 * NB * 4;
        total = g + static_cast<size_t>(U) * 8 * NB * 4;
    }
};

// Stage x, compute g [U][8 NB] of this CTA's units into gs, and meet the peer at a cluster barrier
// (after which both halves of the tile's g may be read). Every thread of the CTA calls it.
template <int NB, int T>
__device__ __forceinline__ void small_gate_phase(const __nv_bfloat16* __restrict__ x,
                                                 const __nv_bfloat16* __restrict__ Wg, int N, int d, int f,
                                                 int tile, int rank, const SmallGateLayout& L, uint8_t* smem,
                                                 cooperative_groups::cluster_group& cluster)
{
    constexpr int U = T / 2;              // hidden units per CTA
    constexpr int MB = U / 16;            // 16-unit blocks per CTA
    constexpr int KS = kSmallWarps / MB;  // warps sharing a block (split of d_model)
    constexpr int NTOK = 8 * NB;
    uint8_t* xs = smem + L.x;
    float* part = reinterpret_cast<float*>(smem + L.part);  // [KS][U][NTOK]
    float* gs = reinterpret_cast<float*>(smem + L.g);       // [U][NTOK]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;

    // the spans past the first batch of every warp (columns 4 KS * 64 .. d of the CTA's rows) move
    // from HBM to L2 while the first batch is loaded and used
    const int pf0 = 4 * KS * 64;
    if (pf0 < d) {
        for (int r = threadIdx.x; r < U; r += blockDim.x) {
            const int u = tile * T + rank * U + r;
            if (u < f) bulk_prefetch_l2(Wg + static_cast<size_t>(u) * d + pf0, static_cast<uint32_t>(d - pf0) * 2u);
        }
    }
    // x rows (zeros past N) by asynchronous copies, in flight with the first weight loads below
    const int chunks = d / 8;
    for (int i = threadIdx.x; i < NTOK * chunks; i += blockDim.x) {
        const int r = i / chunks, c = i - r * chunks;
        const bool in = r < N;
        const size_t src = in ? static_cast<size_t>(r) * d + c * 8 : 0;
        small_cp_async16(xs + r * L.x_stride + c * 16, x + src, in ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");

    const int mb = warp % MB, ks = warp / MB;
    const int ua = tile * T + rank * U + mb * 16 + g, ub = ua + 8;  // this lane's two units
    const bool oka = ua < f, okb = ub < f;
    const __nv_bfloat16* wa = Wg + static_cast<size_t>(oka ? ua : 0) * d + 16 * t;
    const __nv_bfloat16* wb = Wg + static_cast<size_t>(okb ? ub : 0) * d + 16 * t;
    const uint8_t* xg = xs + g * L.x_stride + 32 * t;
    float acc[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = acc[b][2] = acc[b][3] = 0.0f;
    const int nspan = d / 64;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    uint4 w[4][4];  // per span: unit a elements 0-7, 8-15; unit b elements 0-7, 8-15
    auto load_spans = [&](int s0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = s0 + i * KS;
            const bool in = s < nspan;
            w[i][0] = (in && oka) ? ldg_stream16(wa + s * 64) : z;
            w[i][1] = (in && oka) ? ldg_stream16(wa + s * 64 + 8) : z;
            w[i][2] = (in && okb) ? ldg_stream16(wb + s * 64) : z;
            w[i][3] = (in && okb) ? ldg_stream16(wb + s * 64 + 8) : z;
        }
    };
    load_spans(ks);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();  // x staged
    for (int s0 = ks; s0 < nspan; s0 += 4 * KS) {
        if (s0 != ks) load_spans(s0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = s0 + i * KS;
            if (s >= nspan) break;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const uint8_t* xp = xg + b * 8 * L.x_stride + s * 128;
                const uint4 x0 = *reinterpret_cast<const uint4*>(xp);
                const uint4 x1 = *reinterpret_cast<const uint4*>(xp + 16);
                // k step q of the span uses words 2q, 2q + 1 of each lane's 32 bytes
                mma_bf16(acc[b], w[i][0].x, w[i][2].x, w[i][0].y, w[i][2].y, x0.x, x0.y);
                mma_bf16(acc[b], w[i][0].z, w[i][2].z, w[i][0].w, w[i][2].w, x0.z, x0.w);
                mma_bf16(acc[b], w[i][1].x, w[i][3].x, w[i][1].y, w[i][3].y, x1.x, x1.y);
                mma_bf16(acc[b], w[i][1].z, w[i][3].z, w[i][1].w, w[i][3].w, x1.z, x1.w);
            }
        }
    }
    // fragment: (unit g, tokens 2t, 2t+1), (unit g + 8, tokens 2t, 2t+1) of block b
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float* pa = part + (static_cast<size_t>(ks) * U + mb * 16 + g) * NTOK + b * 8 + 2 * t;
        pa[0] = acc[b][0];
        pa[1] = acc[b][1];
        pa[8 * NTOK] = acc[b][2];
        pa[8 * NTOK + 1] = acc[b][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < U * NTOK; i += blockDim.x) {
        float v = part[i];
        for (int k = 1; k < KS; ++k) v += part[static_cast<size_t>(k) * U * NTOK + i];
        gs[i] = v;
    }
    cluster.sync();  // both halves of the tile's g are in shared memory
}

// Pack: warp w of CTA c takes token c + 2 w over the whole tile (the peer's half read from its
// shared memory). The caller keeps both CTAs alive (a second cluster barrier) until this is done.
template <int NB, int T>
__device__ __forceinline__ void small_pack_phase(int N, int f, int nt, int tile, int rank, const SmallGateLayout& L,
                                                 uint8_t* smem, cooperative_groups::cluster_group& cluster,
                                                 int vals_f32, void* __restrict__ vals, uint8_t* __restrict__ idx,
                                                 uint16_t* __restrict__ cnt)
{
    constexpr int U = T / 2;
    constexpr int NTOK = 8 * NB;
    float* gs = reinterpret_cast<float*>(smem + L.g);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = rank + 2 * warp;
    if (warp < NTOK / 2 && r < N) {
        const float* half[2] = {cluster.map_shared_rank(gs, 0), cluster.map_shared_rank(gs, 1)};
        const size_t slot = (static_cast<size_t>(r) * nt + tile) * T;
        int c = 0;
#pragma unroll
        for (int k0 = 0; k0 < T; k0 += 32) {
            const int k = k0 + lane;
            const float v = half[k / U][(k % U) * NTOK + r];
            const bool keep = tile * T + k < f && v > 0.0f;
            const unsigned m = __ballot_sync(0xffffffffu, keep);
            const int pos = c + __popc(m & ((1u << lane) - 1u));
            if (keep) {
                if (vals_f32) static_cast<float*>(vals)[slot + pos] = v;
                else static_cast<__nv_bfloat16*>(vals)[slot + pos] = __float2bfloat16_rn(v);
                idx[slot + pos] = static_cast<uint8_t>(k);
            }
            c += __popc(m);
        }
        if (lane == 0) cnt[static_cast<size_t>(r) * nt + tile] = static_cast<uint16_t>(c);
    }
}

}  // namespace twell
