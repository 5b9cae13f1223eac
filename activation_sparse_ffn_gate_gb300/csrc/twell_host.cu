// twell_host.cu -- host-side services of the C ABI: device info cache, TMA descriptor encoding
// (driver entry point fetched at run time, so the library does not link libcuda), sizes,
// status reporting.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "twell_common.cuh"

namespace twell_host {

namespace {
std::mutex g_mu;
DevInfo g_info[64];
bool g_have[64] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

twell_status dev_info(DevInfo* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TWELL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_have[dev]) {
        DevInfo d{};
        d.device = dev;
        int v = 0;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TWELL_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return TWELL_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return TWELL_ERR_CUDA;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return TWELL_ERR_CUDA;
        d.max_smem_optin = static_cast<size_t>(v);
        g_info[dev] = d;
        g_have[dev] = true;
    }
    *out = g_info[dev];
    return TWELL_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

twell_status make_tmap_bf16(CUtensorMap* out, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                            uint32_t box_inner, uint32_t box_outer)
{
    auto enc = encoder();
    if (enc == nullptr) return TWELL_ERR_CUDA;
    if (!aligned16(base) || (ld * 2) % 16 != 0 || inner == 0 || outer == 0) return TWELL_ERR_INVALID;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TWELL_OK : TWELL_ERR_CUDA;
}

uint64_t wait_limit_ns()
{
    static uint64_t lim = [] {
        const char* s = std::getenv("TWELL_WAIT_LIMIT_MS");
        long v = s ? std::strtol(s, nullptr, 10) : 0;
        return static_cast<uint64_t>(v > 0 ? v : 2000) * 1000000ull;
    }();
    return lim;
}

}  // namespace twell_host

// ------------------------------------------------------------------------------------------------
// C ABI: sizes and status

extern "C" {

size_t twell_packed_vals_bytes(int32_t n_rows, int32_t n_cols, int32_t tile, twell_dtype dtype)
{
    if (n_rows < 0 || n_cols <= 0 || tile <= 0) return 0;
    const size_t nt = (static_cast<size_t>(n_cols) + tile - 1) / tile;
    return static_cast<size_t>(n_rows) * nt * tile * (dtype == TWELL_F32 ? 4 : 2);
}

size_t twell_packed_idx_bytes(int32_t n_rows, int32_t n_cols, int32_t tile)
{
    if (n_rows < 0 || n_cols <= 0 || tile <= 0) return 0;
    const size_t nt = (static_cast<size_t>(n_cols) + tile - 1) / tile;
    return static_cast<size_t>(n_rows) * nt * tile;
}

size_t twell_packed_cnt_bytes(int32_t n_rows, int32_t n_cols, int32_t tile)
{
    if (n_rows < 0 || n_cols <= 0 || tile <= 0) return 0;
    const size_t nt = (static_cast<size_t>(n_cols) + tile - 1) / tile;
    return static_cast<size_t>(n_rows) * nt * 2;
}

twell_status twell_read_status(const int32_t* dev_status, void* stream)
{
    if (dev_status == nullptr) return TWELL_ERR_INVALID;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TWELL_ERR_CUDA;
    int32_t h = 0;
    if (cudaMemcpy(&h, dev_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return TWELL_ERR_CUDA;
    return static_cast<twell_status>(h);
}

const char* twell_status_string(twell_status s)
{
    switch (s) {
    case TWELL_OK: return "ok";
    case TWELL_ERR_INVALID: return "invalid argument";
    case TWELL_ERR_UNSUPPORTED: return "unsupported configuration";
    case TWELL_ERR_BACKUP_FULL: return "hybrid backup buffer full";
    case TWELL_ERR_TIMEOUT: return "bounded device wait timed out";
    case TWELL_ERR_DEVICE_CHECK: return "device-side check failed";
    case TWELL_ERR_CUDA: return "CUDA error";
    case TWELL_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

twell_status twell_device_info(int32_t* sm_count, int32_t* cc_major, int32_t* cc_minor)
{
    twell_host::DevInfo d;
    if (twell_host::dev_info(&d) != TWELL_OK) return TWELL_ERR_CUDA;
    if (sm_count) *sm_count = d.sm_count;
    if (cc_major) *cc_major = d.cc_major;
    if (cc_minor) *cc_minor = d.cc_minor;
    return TWELL_OK;
}

}  // extern "C"
