// twell_common.cuh -- shared device helpers of the sm_103a TwELL library: inline-PTX wrappers for
// mbarriers, TMA (cp.async.bulk.tensor), tcgen05 (TMEM alloc, MMA, commit, loads), bounded waits,
// and host-side launch/validation helpers. Nothing here is specific to one kernel.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only; the driver entry point is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "twell.h"

namespace twell {

// --------------------------------------------------------------------------------------------
// Element helpers

template <typename E>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPer16B = 8;
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};
template <>
struct Elem<float> {
    static constexpr int kPer16B = 4;
    __device__ __forceinline__ static float to_f(float v) { return v; }
    __device__ __forceinline__ static float from_f(float v) { return v; }
};

// Unpack a 16-byte vector of E into fp32.
__device__ __forceinline__ void unpack16(const uint4& v, float (&o)[8], __nv_bfloat16*)
{
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(p[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void unpack16(const uint4& v, float (&o)[4], float*)
{
    o[0] = __uint_as_float(v.x);
    o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z);
    o[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ uint4 pack16(const float (&o)[8], __nv_bfloat16*)
{
    uint4 v;
    __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
    return v;
}
__device__ __forceinline__ uint4 pack16(const float (&o)[4], float*)
{
    return make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                      __float_as_uint(o[3]));
}

// Read-only 16-byte load that does not allocate in L1 (weights are streamed from L2).
__device__ __forceinline__ uint4 ldg_stream16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// --------------------------------------------------------------------------------------------
// Device status

__device__ __forceinline__ void report(int32_t* status, int32_t code)
{
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// --------------------------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of phase completion (for phases known or likely to be complete).
__device__ __forceinline__ bool mbar_test_now(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase of `bar` with parity `parity` has completed. Every wait is bounded: it
// gives up when the CTA-wide abort flag is raised by another thread, or after `limit_ns`, in
// which case it raises the flag and records TWELL_ERR_TIMEOUT in *status. Returns false when
// it gave up.
// Cluster-scope acquire: for phases completed by arrivals from another CTA of the cluster.
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test, suspending the thread in hardware for up to `hint_ns` while the phase is open.
__device__ __forceinline__ bool mbar_test_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

template <bool CLUSTER = false, uint32_t SUSPEND_NS = 0>
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             int32_t* status, uint64_t limit_ns)
{
    const uint32_t a = smem_u32(bar);
    if (!CLUSTER && mbar_test_now(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (CLUSTER ? mbar_test_cluster(a, parity)
                    : (SUSPEND_NS ? mbar_test_suspend(a, parity, SUSPEND_NS) : mbar_test(a, parity)))
            return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            if (abort_flag != nullptr) *abort_flag = 1;
            report(status, TWELL_ERR_TIMEOUT);
            return false;
        }
    }
}

// --------------------------------------------------------------------------------------------
// TMA (tiled tensor copies, global -> shared, completion counted on an mbarrier)

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* tm, int32_t c0, int32_t c1,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// The same copy for a CTA pair (tcgen05 cta_group::2): the completion is counted on the
// mbarrier at shared::cluster address `bar_cluster`, which may be in the peer CTA.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* tm, int32_t c0, int32_t c1,
                                                 uint32_t bar_cluster)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(tm), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
// shared::cluster address of the variable at shared address `smem_addr` in the CTA of `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t smem_addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
// Arrive once on an mbarrier of any CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Bulk (non-tensor) copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from global
// to shared memory, completion counted on `bar`, with an L2 eviction-priority hint.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// Start bringing `bytes` (multiple of 16, 16-byte aligned) of global memory into L2 (no completion
// to wait for): a row needed a little later then comes from L2 instead of HBM.
// First statement of a kernel launched as a programmatic dependent (launch_dep): the kernel after it
// may be scheduled now, and this one waits until the kernel before it has completed and its writes
// are visible. In a kernel launched without the attribute both are no-ops.
__device__ __forceinline__ void pdl_begin()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Barrier over the first `nthreads` threads of the CTA (named barrier `id`, id > 0), returning
// whether any participating thread passed `pred` = true.
__device__ __forceinline__ bool bar_or(int id, int nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Streaming 16-byte store (evict-first in L2).
__device__ __forceinline__ void st_stream16(void* p, const uint4& v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// Two fp32 values, streaming (written once, not read again soon: first to leave L2).
__device__ __forceinline__ void st_stream8(void* p, float a, float b)
{
    asm volatile("st.global.cs.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(a), "f"(b) : "memory");
}
// Read-only 16-byte load, not allocated in L1, with an L2 eviction policy (createpolicy).
__device__ __forceinline__ uint4 ldg_l2hint16(const void* p, uint64_t policy)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

// --------------------------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)

// CG = 1: one CTA; CG = 2: a CTA pair of a cluster (ranks 2i, 2i+1), where one warp of each CTA
// takes part in alloc / relinquish / dealloc. Every tcgen05 instruction of a kernel uses one CG.
template <int CG = 1>
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                     "r"(ncols)
                     : "memory");
}
template <int CG = 1>
__device__ __forceinline__ void tmem_relinquish()
{
    if constexpr (CG == 1) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int CG = 1>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 x bf16 -> fp32). CG = 1: one CTA;
// CG = 2: issued by one thread of the even CTA of a pair, A's M rows and B's N columns split in
// halves between the two CTAs' shared memory (same offsets), D's rows split between their TMEM.
template <int CG = 1>
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    if constexpr (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}
// Arrive once on `bar` when all tcgen05 operations issued so far by this thread have completed.
template <int CG = 1>
__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(bar))
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(bar))
                     : "memory");
}
// The same, arriving on the mbarrier at `bar`'s offset in every CTA of `cta_mask`.
template <int CG = 1>
__device__ __forceinline__ void tc_commit_mc(uint64_t* bar, uint16_t cta_mask)
{
    if constexpr (CG == 1)
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
            ::"r"(smem_u32(bar)), "h"(cta_mask)
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
            ::"r"(smem_u32(bar)), "h"(cta_mask)
            : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptors for tcgen05 with the 128-byte swizzle that TMA writes.
//   bits 0-13 start address >> 4, 16-29 leading byte offset >> 4, 32-45 stride byte offset >> 4,
//   bits 46-48 fixed 0b001, 49-51 base offset (0: tiles are 1024-byte aligned), 61-63 swizzle (2 = 128B).
// K-major operand: rows of 128 B (64 bf16 of K), 8-row swizzle atoms 1024 B apart (SBO); the
// leading offset is not used by this layout. MN-major operand: rows of 128 B (64 bf16 of M or N)
// for one k, 8-row atoms along K 1024 B apart (SBO), 64-element blocks along M/N `lbo` apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo_bytes)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>(1024u >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, A/B major-ness, N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// The same with A and B fp16 (format field 0).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace twell

// --------------------------------------------------------------------------------------------
// Host helpers (defined in twell_host.cu)

namespace twell_host {
// Device properties of the current device (cached per device).
struct DevInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    size_t max_smem_optin;
};
twell_status dev_info(DevInfo* out);

// Bytes of the workspace twell_ffn_fused_fwd needs for N token rows, d_model d, d_ff f (twell_ffn.cu).
size_t fused_ws_bytes(int N, int d, int f);
// Bytes of the workspace twell_ffn_union_fwd needs (twell_union.cu).
size_t union_ws_bytes(int N, int d, int f);
size_t gate_union_ws_bytes(int N, int d, int f);
// The union path for batches of at most kTransposedMaxN tokens, weights on the M side of the products
// (twell_union_small.cu): gate + up with the TwELL pack and h = a * u into H [N, ldo] (fp16), and
// the down product y = H Wd16t_s^T (f_pad = fp, a multiple of 64) split along K over a cluster,
// whose fp32 partials are added in a fixed order in distributed shared memory.
// With Wu_s == nullptr gate_up_small packs the TwELL only (the walk path's gate; H unused).
constexpr int kTransposedMaxN = 128;
constexpr int kDownSmallMaxN = 512;  // down_small serves this many tokens, in 128-token tiles above 128
twell_status gate_up_small(const void* x, const void* Wg_s, const void* Wu_s, int N, int d, int f, int T,
                           const twell_packed* out, __half* H, int ldo, int32_t* dev_status, cudaStream_t s);
twell_status down_small(const __half* H, const void* Wd16t_s, int N, int d, int f, int fp, void* y,
                        int32_t* dev_status, cudaStream_t s);
// Bytes of the workspace twell_ffn_tile_union_fwd needs (twell_tile_union.cu).
size_t tile_union_ws_bytes(int N, int f);
// Bytes of the workspace twell_ffn_decode needs (twell_decode.cu).
size_t decode_ws_bytes(int N, int d, int f, int T);

// 2-D tensor map over a row-major matrix of 16-bit elements: `inner` contiguous elements per row,
// `outer` rows, row pitch `ld` elements; box [box_inner, box_outer]; 128-byte swizzle; zero fill
// out of bounds.
twell_status make_tmap_bf16(CUtensorMap* out, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                            uint32_t box_inner, uint32_t box_outer);

// Limit of every bounded device-side wait, in ns (TWELL_WAIT_LIMIT_MS in the environment, else 2 s).
uint64_t wait_limit_ns();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline twell_status launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

// Launch `kern` as a programmatic dependent of the kernel before it on `s`; the kernel must begin
// with twell::pdl_begin() (its first statement), so that it reads and writes nothing before the
// previous kernel has completed.
template <typename... KArgs, typename... Args>
twell_status launch_dep(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...) == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}
}  // namespace twell_host

namespace twell_host {
// Validate a TwELL descriptor against the expected shape and element type.
// Data pointers may be null only for an empty matrix (N == 0).
inline twell_status check_packed(const twell_packed* p, int32_t N, int32_t f, int32_t T, twell_dtype dt)
{
    if (p == nullptr) return TWELL_ERR_INVALID;
    if (p->n_rows != N || p->n_cols != f || p->tile != T || p->cap != T || p->dtype != dt) return TWELL_ERR_INVALID;
    if (T != 64 && T != 128 && T != 256) return TWELL_ERR_UNSUPPORTED;
    if (N == 0) return TWELL_OK;
    if (p->vals == nullptr || p->idx == nullptr || p->cnt == nullptr) return TWELL_ERR_INVALID;
    if (!aligned16(p->vals) || !aligned16(p->idx) || !aligned16(p->cnt)) return TWELL_ERR_INVALID;
    return TWELL_OK;
}
inline bool dtype_ok(twell_dtype dt) { return dt == TWELL_BF16 || dt == TWELL_F32; }

// TwELL pack of a bf16 gate matrix into a TwELL with fp32 values (exact widening; twell_pack.cu).
twell_status pack_gate_widened(const void* G, int N, int f, const twell_packed* out, int32_t* status, cudaStream_t s);
}  // namespace twell_host
