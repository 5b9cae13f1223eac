// twell_hybrid.cu -- hybrid-format training forward and backward (in progress).
#include "twell_common.cuh"

extern "C" size_t twell_workspace_bytes(twell_op op, int32_t N, int32_t d, int32_t f, int32_t tile, int32_t K,
                                        int32_t backup_cap)
{
    (void)op; (void)N; (void)d; (void)f; (void)tile; (void)K; (void)backup_cap;
    return 0;
}

extern "C" twell_status twell_hybrid_fwd(const void*, const void*, const void*, const void*, int32_t, int32_t, int32_t,
                                         int32_t, float, twell_dtype, const twell_hybrid*, void*, void*, size_t, void*)
{
    return TWELL_ERR_UNSUPPORTED;
}

extern "C" twell_status twell_hybrid_bwd(const void*, const void*, const void*, const void*, const twell_hybrid*,
                                         const void*, int32_t, int32_t, int32_t, float, void*, float*, float*, float*,
                                         void*, size_t, void*)
{
    return TWELL_ERR_UNSUPPORTED;
}

extern "C" twell_status twell_hybrid_route_from_gate(const void*, int32_t, int32_t, int32_t, twell_dtype,
                                                     const twell_hybrid*, void*, size_t, void*)
{
    return TWELL_ERR_UNSUPPORTED;
}
