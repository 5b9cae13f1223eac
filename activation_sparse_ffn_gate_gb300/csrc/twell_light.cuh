// twell_light.cuh -- host side of the tensor-core kernels for the light rows of the hybrid
// training format (twell_light.cu).
#pragma once

#include "twell_common.cuh"

namespace twell_host {

// Forward of the light rows: for every row r with hcnt[r] <= K (0xFFFF marks a backup row, which
// is skipped) and each kept entry e = r*K + k (k < hcnt[r]) of column j = hcol[e], a = ha[e]:
// u = x_r . Wu_s[j] (stored in hu[e]; slots k >= hcnt[r] get 0), h = a u, y_r = sum h Wd_s[j]
// (bf16; 0 for a row without entries), and sum |h| added to *l1acc. d must be 512, 1024, 2048 or
// 2560, else TWELL_ERR_UNSUPPORTED and nothing is launched. `tickets`: one int of workspace,
// cleared on the stream by the call.
twell_status light_fwd_bulk(const void* x, const void* Wu_s, const void* Wd_s, int N, int d, int f, int K,
                            const float* ha, const uint16_t* hcol, const uint16_t* hcnt, float* hu, void* y,
                            double* l1acc, int* tickets, int32_t* status, cudaStream_t s);

// Backward of the light rows: per kept entry dh = dy_r . Wd_s[j], g = dh + l1_scale sgn(h) with
// h = a u, du = g a, dg = g u, ent[3e .. 3e+2] = {h, du, dg}, and dx_r = sum du Wu_s[j] + dg Wg_s[j]
// (fp32; 0 for a light row without entries; backup rows untouched). Same shapes as the forward.
twell_status light_bwd_bulk(const void* dy, const void* Wg_s, const void* Wu_s, const void* Wd_s, int N, int d,
                            int f, int K, const float* ha, const float* hu, const uint16_t* hcol,
                            const uint16_t* hcnt, float l1_scale, float* ent, float* dx, int* tickets,
                            int32_t* status, cudaStream_t s);

}  // namespace twell_host
