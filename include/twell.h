/*
 * twell.h -- C ABI of the GB300 (sm_103a) activation-sparse gated FFN library (libtwell_gb300.so).
 *
 * The layer is  y = (ReLU(x Wg) * (x Wu)) Wd  with the gate activation kept in the tile-wise
 * ELL (TwELL) format. Passages that define each operation are cited by page title and section:
 *   [AIM] aimodeling.com news item "TwELL：Sakana AI与NVIDIA联合提出稀疏LLM推理加速20%，解决GPU批处理落地难题",
 *         summary paragraph n (¶n).
 *   [TG]  Telegram post "Sakana AI и NVIDIA представили TwELL ..." (ai_machinelearning_big_data),
 *         sections "Вот тут и решает TwELL", "Инференс", "Обучение".
 *   [PUL] pulsen.vercel.app "Sakana AI og NVIDIA introduserer TwELL ...", paragraph n.
 *   [TC]  Tencent Cloud "一文读懂 NVIDIA 与 Sakana AI 联手打造的稀疏 LLM 黑科技", sections 1-6.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Shapes: N tokens, d = d_model, f = d_ff, T = TwELL tile width, nt = ceil(f / T),
 *   K = hybrid per-row capacity.
 * - Weights are stored one row per hidden unit ("rows of Wu and Wd", [TG] "Инференс"):
 *   Wg_s = Wg^T, Wu_s = Wu^T and Wd_s = Wd are all [f, d] row-major. x, y, dy, dx are [N, d]
 *   row-major. So G = x Wg_s^T, U = x Wu_s^T, y = (ReLU(G) * U) Wd_s.
 * - Every pointer argument named as device memory must be device memory allocated by the
 *   caller; the library never allocates, never frees and keeps no pointer after a call returns.
 *   Struct arguments (twell_packed, twell_hybrid) are host structs that hold device pointers.
 * - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *   default stream). Outputs are valid once the stream reaches the call.
 * - Alignment: every device pointer must be 16-byte aligned; d must be a multiple of 8.
 * - Element type: TWELL_BF16 (bf16 storage, fp32 accumulation, tcgen05 tensor cores for the
 *   gate) or TWELL_F32 (fp32 storage and arithmetic on CUDA cores; small layers and tests).
 * - Errors: argument errors are detected on the host and returned before anything is launched
 *   (nothing is written). Conditions found on the device (a bounded wait that ran out, a
 *   failed device-side check, a full backup buffer) are written to *dev_status (one int32 in
 *   device memory, first error wins, never cleared by the library) as a twell_status code; read
 *   it with twell_read_status(). Launch failures return TWELL_ERR_CUDA.
 */
#ifndef TWELL_GB300_H
#define TWELL_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TWELL_API __attribute__((visibility("default")))
#else
#define TWELL_API
#endif

typedef enum {
    TWELL_OK = 0,
    TWELL_ERR_INVALID = 1,     /* bad argument (null pointer, size, alignment, mismatch) */
    TWELL_ERR_UNSUPPORTED = 2, /* valid but not supported here (dtype, tile width, device) */
    TWELL_ERR_BACKUP_FULL = 3, /* hybrid: more overflow rows than backup_cap (device-reported) */
    TWELL_ERR_TIMEOUT = 4,     /* a bounded device-side wait ran out (device-reported) */
    TWELL_ERR_DEVICE_CHECK = 5,/* a device-side consistency check failed (device-reported) */
    TWELL_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
    TWELL_ERR_WORKSPACE = 7    /* workspace missing or smaller than twell_workspace_bytes() */
} twell_status;

typedef enum { TWELL_BF16 = 0, TWELL_F32 = 1 } twell_dtype;

typedef enum {
    TWELL_OP_GATE_PACK = 0,
    TWELL_OP_FFN_FUSED_FWD = 1,
    TWELL_OP_HYBRID_FWD = 2,
    TWELL_OP_HYBRID_BWD = 3,
    TWELL_OP_HYBRID_ROUTE = 4,
    TWELL_OP_FFN_UNION_FWD = 5,
    TWELL_OP_FFN_DECODE = 6,
    TWELL_OP_FFN_TILE_UNION_FWD = 7,
    TWELL_OP_FFN_GATE_UNION_FWD = 8
} twell_op;

/* A TwELL matrix of gate activations a = ReLU(G), [n_rows, n_cols] ([TG] "Вот тут и решает TwELL";
 * [TC] §2). The columns are cut into nt = ceil(n_cols / tile) tiles of `tile` columns (the last
 * one partial when tile does not divide n_cols). For row r and tile t:
 *   cnt[r*nt + t]                 number of kept entries (g > 0) of that row in that tile;
 *   vals[(r*nt + t)*cap + k]      value of the k-th kept entry, k < cnt (element type `dtype`);
 *   idx [(r*nt + t)*cap + k]      its column inside the tile (0..tile-1), strictly ascending in k.
 * Slots k >= cnt are never written or read. cap must equal tile (lossless: a tile can never
 * overflow). tile is 64, 128 or 256. All three arrays are caller-owned device memory. */
typedef struct {
    int32_t n_rows;
    int32_t n_cols;
    int32_t tile;
    int32_t cap;
    twell_dtype dtype;
    void* vals;
    uint8_t* idx;
    uint16_t* cnt;
} twell_packed;

/* The hybrid training format ([TG] "Обучение"; [TC] §3): each row either fits in one
 * globally aligned sparse block of fixed capacity K or, when it has more than K nonzeros,
 * goes to a dense backup buffer. All pointers are caller-owned device memory.
 *   cnt[n_rows]          uint16: nonzeros of a light row (<= K), or 0xFFFF for a backup row;
 *   col[n_rows*K]        uint16: light rows' kept columns in ascending order (slots >= cnt: 0);
 *   a  [n_rows*K]        fp32: a = ReLU(g) at those columns (slots >= cnt: +0);
 *   u  [n_rows*K]        fp32: u = x Wu_s^T at those columns (filled by hybrid_fwd);
 *   backup_rows[backup_cap]  int32: backup row indices in ascending order;
 *   n_backup[1]          int32: number of overflow rows (may exceed backup_cap: then the call
 *                        reports TWELL_ERR_BACKUP_FULL, only backup_cap rows are stored and the
 *                        outputs of the other overflow rows are undefined);
 *   A_b[backup_cap*n_cols]   fp32: dense a rows of the backup rows;
 *   U_b[backup_cap*n_cols]   fp32: dense u rows of the backup rows (filled by hybrid_fwd);
 *   l1[1]                fp32: L1 term lambda * mean|h| (filled by hybrid_fwd);
 *   dev_status[1]        int32 device status word (see the conventions above).
 * Rows of a light row that are not written are never read; a row is in exactly one of the sparse
 * block and the backup. dtype must be TWELL_BF16 (the element type of x, weights, y, dy, dx). */
typedef struct {
    int32_t n_rows;
    int32_t n_cols;
    int32_t K;
    int32_t backup_cap;
    twell_dtype dtype;
    void* a;
    void* u;
    uint16_t* col;
    uint16_t* cnt;
    int32_t* backup_rows;
    int32_t* n_backup;
    void* A_b;
    void* U_b;
    float* l1;
    int32_t* dev_status;
} twell_hybrid;

/* ------------------------------------------------------------------------------------------
 * Sizes. Bytes of the three TwELL arrays for [n_rows, n_cols] with tile width `tile`
 * (cap = tile), and workspace bytes an operation needs (0 = none; then ws may be NULL).
 * Return 0 on invalid arguments.
 */
TWELL_API size_t twell_packed_vals_bytes(int32_t n_rows, int32_t n_cols, int32_t tile, twell_dtype dtype);
TWELL_API size_t twell_packed_idx_bytes(int32_t n_rows, int32_t n_cols, int32_t tile);
TWELL_API size_t twell_packed_cnt_bytes(int32_t n_rows, int32_t n_cols, int32_t tile);
TWELL_API size_t twell_workspace_bytes(twell_op op, int32_t N, int32_t d, int32_t f, int32_t tile, int32_t K,
                             int32_t backup_cap);

/* ------------------------------------------------------------------------------------------
 * Gate projection with the TwELL pack in its epilogue ([AIM] ¶3; [TG] "Вот тут и решает TwELL";
 * [PUL] ¶3; [TC] §2): G = x Wg_s^T accumulated in fp32, and in the same kernel, per token row
 * and column tile, a = ReLU(G) is packed as values + in-tile indices + count. A gate entry is
 * kept iff its fp32 accumulator is > 0. No dense G is written. x [N, d], Wg_s [f, d] (device,
 * element type `dtype`). `out` must describe an [N, f] TwELL matrix with out->tile = T; its
 * values are stored in out->dtype: TWELL_F32 keeps the fp32 accumulator exactly (allowed for
 * both input types), TWELL_BF16 rounds it to nearest even (bf16 inputs only).
 * ws/ws_bytes: workspace (twell_workspace_bytes(TWELL_OP_GATE_PACK, ...), currently 0).
 */
TWELL_API twell_status twell_gate_pack(const void* x, const void* Wg_s, int32_t N, int32_t d, int32_t f,
                             int32_t T, twell_dtype dtype, const twell_packed* out, void* ws,
                             size_t ws_bytes, int32_t* dev_status, void* stream);

/* Fused up+down projection over a TwELL matrix ([AIM] ¶3; [TG] "Инференс"; [PUL] ¶3; [TC] §2):
 * for every token row, walk only its packed nonzeros (column j, value a), gather row j of Wu_s
 * and of Wd_s, and accumulate y_r += a * (x_r . Wu_s[j]) * Wd_s[j] in fp32; y is stored in the
 * TwELL's dtype. The hidden activation h is never written to memory. Rows with no nonzeros get
 * y = 0. x [N, d], Wu_s / Wd_s [f, d], y [N, d] (device, element type `dtype`; the TwELL
 * values may be bf16 or fp32 independently, except that fp32 inputs need fp32 values).
 * d <= 8192 (bf16) / 4096 (fp32); f / tile <= 1024 tiles.
 * ws/ws_bytes: device workspace of at least twell_workspace_bytes(TWELL_OP_FFN_FUSED_FWD, N, d,
 * ...) bytes, 16-byte aligned, required when N > 0 (else TWELL_ERR_WORKSPACE). It holds the work
 * counter the kernel hands out rows from, a work plan (rows above 128 nonzeros are cut into items
 * of at most 128, walked by different warps, and their fp32 partial rows are added up in item
 * order by the last one to finish; the other rows are handed out longest class first) and those
 * partial rows: about 12 B per row plus N/8 (64 .. 4096) partial rows of 4*d bytes. The call
 * clears its header on `stream`, so two calls in flight at the same time must not share one
 * workspace. Its contents need not be initialised. y is the same bit for bit from call to call,
 * unless more rows want splitting than the N/8 item slots hold (those that find no room are
 * walked whole, and which ones those are depends on scheduling).
 * A corrupt TwELL (count above the tile width, in-tile index >= tile, column >= f) is reported
 * as TWELL_ERR_DEVICE_CHECK in *dev_status; such entries contribute nothing.
 */
TWELL_API twell_status twell_ffn_fused_fwd(const void* x, const void* Wu_s, const void* Wd_s,
                                 const twell_packed* a, int32_t N, int32_t d, int32_t f,
                                 twell_dtype dtype, void* y, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, void* stream);

/* twell_ffn_fused_fwd with the down projection in fp16: Wd16_s is Wd_s converted once to fp16
 * (twell_convert_f16; the conversion is exact for every bf16 weight in [2^-17, 65504] in
 * magnitude, and loses no more than 2^-25 in absolute terms below that), and each h = a * u is
 * rounded once to fp16 (11 significant bits, against ~16 for the bf16 hi + lo pair of
 * twell_ffn_fused_fwd), which halves the tensor-core products of the down projection. Products
 * are accumulated in fp32, as there. bf16 x, Wu_s and y; TwELL values bf16 or fp32; d a multiple
 * of 256 in [512, 3072] (else TWELL_ERR_UNSUPPORTED). Workspace, determinism and error
 * reporting as twell_ffn_fused_fwd.
 */
TWELL_API twell_status twell_ffn_fused_fwd_f16down(const void* x, const void* Wu_s, const void* Wd16_s,
                                         const twell_packed* a, int32_t N, int32_t d, int32_t f,
                                         void* y, void* ws, size_t ws_bytes, int32_t* dev_status,
                                         void* stream);

/* n bf16 values at src to fp16 at dst (device pointers, no overlap), round to nearest even. A
 * finite value beyond the fp16 range is stored as infinity and reported as
 * TWELL_ERR_DEVICE_CHECK in *dev_status.
 */
TWELL_API twell_status twell_convert_f16(const void* src, void* dst, int64_t n, int32_t* dev_status,
                               void* stream);

/* dst [cols, rows] (fp16) = the transpose of src [rows, cols] (bf16, row-major) converted to fp16 with
 * the same rounding and overflow reporting as twell_convert_f16 (e.g. Wd_s [d_ff, d_model] ->
 * Wd16t_s [d_model, d_ff] for twell_ffn_union_fwd). rows <= 2,097,120 (else TWELL_ERR_UNSUPPORTED).
 * Device pointers; asynchronous on `stream`. */
TWELL_API twell_status twell_convert_f16_transposed(const void* src, void* dst, int32_t rows, int32_t cols,
                                                    int32_t* dev_status, void* stream);

/* The whole layer for a batch of at most 16 tokens (decoding) in two launches: the gate + pack of
 * twell_gate_pack (the same TwELL in *a_out, bit for bit) and, in the same kernel, the walk of each
 * column tile's kept entries by the CTAs that computed them ([AIM] ¶3; [TG] "Инференс"; [PUL] ¶3;
 * [TC] §2): the walk is separable by column tile, y_r = sum over tiles of sum over the tile's kept
 * j of a * (x_r . Wu_s[j]) * Wd_s[j]. Each CTA (half a column tile) forms u and h = a * u for its
 * units in fp32 (a as stored in the TwELL), adds h * Wd_s[j] in fp32 over its units in ascending
 * order and stores one fp32 partial row per token; a second kernel adds each token's partial rows
 * in a fixed order and stores y (bf16). y is the same bit for bit from call to call and does not
 * depend on scheduling; it agrees with twell_ffn_fused_fwd on the same TwELL to fp32 summation
 * order. bf16 x, Wg_s, Wu_s, Wd_s, y; 0 <= N <= 16, d_model a multiple of 64 up to 4096, tile 64,
 * 128 or 256 (else TWELL_ERR_UNSUPPORTED); a_out describes an [N, f] TwELL with tile T, values
 * bf16 or fp32. ws: twell_workspace_bytes(TWELL_OP_FFN_DECODE, N, d, f, T, 0, 0) bytes (a flag
 * and an fp32 partial row of d_model per (CTA, token): 2 * ceil(f / T) CTAs), 16-byte aligned,
 * required when N > 0; its contents need not be initialised, and two calls in flight at the same
 * time must not share it.
 */
TWELL_API twell_status twell_ffn_decode(const void* x, const void* Wg_s, const void* Wu_s, const void* Wd_s,
                              int32_t N, int32_t d, int32_t f, int32_t T, const twell_packed* a_out,
                              void* y, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* The same y from the same TwELL for a layer too dense for the walk: with more than a few percent
 * of d_ff kept per token the union of the units a tile of 128 tokens keeps is nearly all of d_ff,
 * so the up and down projections are dense contractions over all of it, on the tensor cores ([TC]
 * §3: tensor cores for the heavy work). Steps: a is written into H [N, f_pad] (fp16, f_pad = f
 * rounded up to 64) at each row's kept columns, with a per-row keep mask; H = (x Wu_s^T) * a
 * (tcgen05 GEMM on SM pairs, the product formed in its epilogue where the mask is set, h stored in
 * place as fp16: 11 significant bits); y = H Wd16_s (tcgen05 GEMM on SM pairs over f_pad, fp16
 * operands, bf16 y). Wd16t_s is the transpose of Wd_s converted once to fp16 ([d, f]:
 * twell_convert_f16_transposed), so that the down GEMM reads both operands K-major. For N <= 512
 * the down product runs transposed (y^T = Wd16t_s H^T, rows of Wd16t_s on the MMA's M side, tokens in
 * tiles of up to 128, K split over a cluster of CTAs whose fp32 partials are added in a fixed order
 * in shared memory).
 * bf16 x, Wu_s, y; d and f multiples of 8; x [N, d], Wu_s [f, d], Wd16t_s [d, f], y [N, d], device,
 * 16-byte aligned. ws: twell_workspace_bytes(TWELL_OP_FFN_UNION_FWD, N, d, f, ...) bytes (H and the
 * masks, 2.125 * N * f_pad bytes), required when N > 0. A corrupt TwELL entry (count above the tile
 * width, column >= f) is reported as TWELL_ERR_DEVICE_CHECK in *dev_status and contributes nothing;
 * so is an a or h beyond the fp16 range.
 */
TWELL_API twell_status twell_ffn_union_fwd(const void* x, const void* Wu_s, const void* Wd16t_s,
                                 const twell_packed* a, int32_t N, int32_t d, int32_t f,
                                 twell_dtype dtype, void* y, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, void* stream);

/* twell_gate_pack followed by twell_ffn_union_fwd, with the gate and the up projection in one
 * tensor-core GEMM: each tile of an SM pair computes g = x Wg_s^T and u = x Wu_s^T for the same 128
 * units (the pair's two CTAs load Wg_s and Wu_s rows respectively, x is shared), and its epilogue
 * packs ReLU(g) into *out -- the TwELL twell_gate_pack writes, bit for bit ([AIM] ¶3, [TC] §2:
 * the pack in the gate GEMM's epilogue) -- and stores h = a * u (a = the packed value; fp16, 11
 * significant bits; 0 where g <= 0) into the workspace; then y = H Wd16_s as in twell_ffn_union_fwd.
 * For N <= 128 both products run transposed, the weights on the MMA's M side and the tokens as its
 * N columns: each CTA stacks 64 units' Wg_s rows over their Wu_s rows, and two CTAs form one
 * 128-unit tile whose TwELL is the same, bit for bit; up to N = 512 the down product runs
 * transposed as in twell_ffn_union_fwd.
 * For layers whose density the walk no longer serves: the union of the units a tile of 128 tokens
 * keeps is then most of d_ff ([TC] §3: tensor cores for the heavy work).
 * bf16 x, Wg_s, Wu_s, y (dtype must be TWELL_BF16); d and f multiples of 8; T = 64 or 128 (else
 * TWELL_ERR_UNSUPPORTED); x [N, d], Wg_s / Wu_s [f, d], Wd16t_s [d, f] (twell_convert_f16_transposed
 * of Wd_s), y [N, d]; *out a TwELL of N rows, f columns, tile T, fp32 or bf16 values. Device
 * pointers, 16-byte aligned. ws: twell_workspace_bytes(TWELL_OP_FFN_GATE_UNION_FWD, N, d, f, ...)
 * bytes (H [N, f_pad] fp16, f_pad = f rounded up to 64), required when N > 0. An h beyond the fp16
 * range is recorded as TWELL_ERR_DEVICE_CHECK in *dev_status.
 */
TWELL_API twell_status twell_ffn_gate_union_fwd(const void* x, const void* Wg_s, const void* Wu_s,
                                      const void* Wd16t_s, int32_t N, int32_t d, int32_t f, int32_t T,
                                      twell_dtype dtype, const twell_packed* out, void* y, void* ws,
                                      size_t ws_bytes, int32_t* dev_status, void* stream);

/* y = (a * (x Wu_s^T)) Wd_s from the TwELL a, as tensor-core GEMMs over the units each tile of
 * 128 tokens keeps -- the tile's union U_m -- with the union's weight rows gathered ([TG] "Инференс":
 * the kernel gathers only the needed rows of Wu and Wd; [TC] §3: tensor cores take the heavy work).
 * Per tile m: H_m[r, p] = a[r, U_m[p]] * (x_r . Wu_s[U_m[p]]) over p < |U_m| (tcgen05, B = gathered
 * Wu_s rows, the product in the epilogue, h stored once as fp16), then y_m = H_m Wd16_s[U_m]
 * (tcgen05 over K = |U_m|, B = gathered rows of Wd16_s). Each weight row is read once per tile of
 * 128 tokens instead of once per token that keeps it. Wd16_s is Wd_s converted to fp16 once
 * (twell_convert_f16: the same values for weights of magnitude 2^-14 .. 65504; smaller ones move by
 * at most 2^-25); h carries 11 significant bits.
 * x [N, d] bf16, Wu_s [f, d] bf16, Wd16_s [f, d] fp16, y [N, d] bf16, all device, 32-byte aligned;
 * d a multiple of 64 (else TWELL_ERR_UNSUPPORTED); f <= 65535; a: any tile width, fp32 or bf16
 * values. ws: twell_workspace_bytes(TWELL_OP_FFN_TILE_UNION_FWD, N, d, f, ...) bytes, 32-byte
 * aligned, required when N > 0 (per tile: the union list and bitmap; H as fp16 [N, f rounded up to
 * 256]); its contents need not be initialised; two calls in flight at the same time must not share
 * it. A corrupt TwELL entry (count above the tile width, in-tile index >= T, column >= f) is
 * recorded as TWELL_ERR_DEVICE_CHECK and contributes nothing; so is an h beyond the fp16 range
 * (|h| >= 65520, stored as infinity).
 */
TWELL_API twell_status twell_ffn_tile_union_fwd(const void* x, const void* Wu_s, const void* Wd16_s,
                                                const twell_packed* a, int32_t N, int32_t d, int32_t f, void* y,
                                                void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Hybrid-format training forward ([TG] "Обучение"; [TC] §3), bf16 only (d_ff a multiple of
 * 64, d_model at most 4096, d_ff at most 65535): gate GEMM + TwELL pack,
 * routing of each row to the sparse block (nnz <= K) or to the dense backup (nnz > K, in
 * ascending row order), the up/down products (gathered rows of Wu_s / Wd_s for light rows,
 * dense tensor-core GEMMs for backup rows), y [N, d], and the L1 term
 * l1_coef * mean|h| over all N*f entries of h ([AIM] ¶4; [PUL] ¶4) into *ctx->l1.
 * ctx describes caller-owned buffers for N = ctx->n_rows, f = ctx->n_cols.
 * ws: at least twell_workspace_bytes(TWELL_OP_HYBRID_FWD, N, d, f, 0, K, backup_cap) bytes.
 */
TWELL_API twell_status twell_hybrid_fwd(const void* x, const void* Wg_s, const void* Wu_s, const void* Wd_s,
                              int32_t N, int32_t d, int32_t f, int32_t K, float l1_coef,
                              twell_dtype dtype, const twell_hybrid* ctx, void* y, void* ws,
                              size_t ws_bytes, void* stream);

/* Hybrid-format training backward ([TG] "Обучение": no product of two dense matrices for the
 * sparse rows), bf16 storage: given the context filled by twell_hybrid_fwd and dy [N, d],
 * computes the gradients of  <y, dy> + l1_coef * mean|h| :
 *   dh = dy_r . Wd_s[j] + l1_coef * sgn(h) / (N f),  du = dh * a,  dg = dh * u  (at kept entries)
 *   dx [N, d] (fp32)          = sum_j du * Wu_s[j] + dg * Wg_s[j]
 *   dWg_s, dWu_s, dWd_s [f, d] (fp32, overwritten) = sum_r dg x_r, du x_r, h dy_r.
 * Gradients are written in fp32: a bf16 copy of dx rounds its largest element by up to 2^-8 of
 * itself, more than the accuracy the layer is held to.
 * Backup rows take dh and dx from dense tensor-core GEMMs; the weight gradients of every kept
 * entry, light or backup, are summed per hidden unit in row order (deterministic). Same shape
 * limits as the forward.
 * ws: at least twell_workspace_bytes(TWELL_OP_HYBRID_BWD, N, d, f, 0, K, backup_cap) bytes; it
 * need not hold anything from the forward call (the context carries what the backward needs).
 */
TWELL_API twell_status twell_hybrid_bwd(const void* x, const void* Wg_s, const void* Wu_s, const void* Wd_s,
                              const twell_hybrid* ctx, const void* dy, int32_t N, int32_t d,
                              int32_t f, float l1_coef, float* dx, float* dWg_s, float* dWu_s,
                              float* dWd_s, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * Dead-column compaction. The pages report that more than 30% of the gate's hidden units never
 * fire once training has settled ([PUL] ¶5). A unit that never fires adds nothing to y, so the
 * layer can run on the live units alone: count, per column, how often a calibration batch's TwELL
 * matrix keeps it (twell_column_activity), gather the rows of Wg_s, Wu_s and Wd_s of the columns
 * that fired (twell_gather_rows), and call twell_gate_pack / twell_ffn_fused_fwd with d_ff = the
 * number of live units. With the live columns kept in ascending order the compacted layer gives
 * the same y, bit for bit, on any batch whose active units are among them. The pages state the
 * observation, not this procedure.
 */

/* *total += the number of kept entries of `a` (the sum of its counts; device uint64, the caller
 * clears it): the batch's density is *total / (n_rows * n_cols), which is what a caller needs to
 * choose between twell_ffn_fused_fwd and twell_ffn_tile_union_fwd for the next batch. A count above
 * the tile width is reported as TWELL_ERR_DEVICE_CHECK and counts as 0. Asynchronous on `stream`. */
TWELL_API twell_status twell_count_nonzeros(const twell_packed* a, unsigned long long* total, int32_t* dev_status,
                                            void* stream);

/* col_counts[j] += the number of rows of `a` that keep column j (device int32 [a->n_cols]; the
 * call adds to what is there, the caller clears it). A bad entry (count above the tile width,
 * in-tile index >= tile, column >= n_cols) is reported as TWELL_ERR_DEVICE_CHECK in *dev_status
 * and skipped. */
TWELL_API twell_status twell_column_activity(const twell_packed* a, int32_t* col_counts, int32_t* dev_status,
                                   void* stream);

/* dst[i, :] = src[rows[i], :] for i < n (device; src [n_src, d], dst [n, d] row-major, element
 * type dtype, d * element size a multiple of 16 bytes, both 16-byte aligned; rows int32 [n]). A
 * row index outside [0, n_src) is reported as TWELL_ERR_DEVICE_CHECK and its output row is 0. */
TWELL_API twell_status twell_gather_rows(const void* src, int32_t n_src, const int32_t* rows, int32_t n,
                               int32_t d, twell_dtype dtype, void* dst, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------------------------
 * Test exports. They run the same device code as the calls above on a gate matrix the caller
 * provides, so packing and routing can be compared bit for bit with an independent reference.
 */

/* Dense [N, f] copy of a TwELL matrix (zeros outside the packed entries), in a->dtype. */
TWELL_API twell_status twell_unpack(const twell_packed* a, void* dense_out, int32_t* dev_status, void* stream);

/* TwELL pack of a given gate matrix G [N, f] (device, dtype): keep g > 0, values copied
 * unchanged. Uses the warp-ballot compaction of the gate epilogue. */
TWELL_API twell_status twell_pack_from_gate(const void* G, int32_t N, int32_t f, int32_t T, twell_dtype dtype,
                                  const twell_packed* out, int32_t* dev_status, void* stream);

/* Hybrid routing of a given gate matrix G [N, f] (device, bf16): the routing kernels of
 * twell_hybrid_fwd applied to pack(G) with tile width 128. Fills ctx->cnt, col, a,
 * backup_rows, n_backup, A_b (not u, U_b, l1). ws: twell_workspace_bytes(TWELL_OP_HYBRID_ROUTE). */
TWELL_API twell_status twell_hybrid_route_from_gate(const void* G, int32_t N, int32_t f, int32_t K,
                                          twell_dtype dtype, const twell_hybrid* ctx, void* ws,
                                          size_t ws_bytes, void* stream);

/* Dense fp32 G = x Wg_s^T [N, f] (row-major, ld = f) from the same tcgen05 mainloop as
 * twell_gate_pack, with a plain store epilogue (bf16 inputs only). */
TWELL_API twell_status twell_gate_gemm(const void* x, const void* Wg_s, int32_t N, int32_t d, int32_t f,
                             float* G_out, int32_t* dev_status, void* stream);

/* Hybrid routing of an already packed TwELL matrix `a` (fp32 values, tile 128, as written by
 * twell_gate_pack or twell_pack_from_gate) into ctx -- the same kernels and the same results as
 * the routing inside twell_hybrid_fwd / twell_hybrid_route_from_gate (ctx->cnt, col, a,
 * backup_rows, n_backup, A_b; not u, U_b, l1) -- without any workspace and without allocating.
 * The pages have no counterpart: this call exists for callers that cannot allocate device memory
 * or pass a workspace (code inside a framework whose caching allocator owns all device memory;
 * plug-in hosts whose interface carries only inputs and outputs; latency-critical loops where an
 * allocation would synchronise the device). ctx->u, ctx->U_b and ctx->l1 are not used and may be
 * null; cnt, n_backup, dev_status, and col and a (K > 0), backup_rows and A_b (backup_cap > 0)
 * are required.
 * Its only scratch, the overflow-row count of each 32-row block, is a fixed array of 32768 int32
 * inside the library: every GPU that loads the library keeps it (128 KB) until the process exits.
 * Limit: a->n_rows <= 1,048,576; larger inputs return TWELL_ERR_UNSUPPORTED before any launch.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress), so make
 * that first call before any stream capture. All calls share the one array: two calls that
 * overlap on the GPU (different streams, no ordering between them) race and give wrong routes;
 * order them on one stream or with events. */
TWELL_API twell_status twell_hybrid_route_noalloc(const twell_packed* a, int32_t K,
                                                  const twell_hybrid* ctx, void* stream);

/* The bounded mbarrier wait every kernel of the library uses, on its own: one warp initialises an
 * mbarrier that expects one arrival and waits on it with a limit of limit_ms milliseconds. With
 * arrive != 0 the warp's lane 0 arrives first and the wait ends at once; with arrive == 0 nothing
 * ever arrives, the wait gives up after limit_ms, records TWELL_ERR_TIMEOUT in *dev_status and
 * the kernel returns, leaving the context usable. This is how failure detection is tested without
 * hanging or faulting a GPU: the limit of the real kernels' waits (TWELL_WAIT_LIMIT_MS, 2 s by
 * default) takes the same path. limit_ms in [1, 10000], else TWELL_ERR_INVALID. */
TWELL_API twell_status twell_wait_probe(int32_t arrive, int32_t limit_ms, int32_t* dev_status, void* stream);

/* C[M, N] = A * B in fp32 from the tcgen05 GEMM used by the hybrid backup rows, bf16 operands:
 * A is [M, K] row-major (a_mn = 0) or [K, M] row-major (a_mn = 1); B is [N, K] row-major
 * (b_mn = 0) or [K, N] row-major (b_mn = 1); C is [M, N] row-major. N and the contiguous
 * extents must be multiples of 8. */
TWELL_API twell_status twell_gemm_test(const void* A, const void* B, int32_t M, int32_t N, int32_t K,
                                       int32_t a_mn, int32_t b_mn, float* C, int32_t* dev_status,
                                       void* stream);

/* ------------------------------------------------------------------------------------------
 * Status.
 */

/* Synchronises `stream`, then returns the code held in *dev_status (TWELL_OK if 0). */
TWELL_API twell_status twell_read_status(const int32_t* dev_status, void* stream);

/* Static text for a status code. */
TWELL_API const char* twell_status_string(twell_status s);

/* Number of SMs and the compute capability of the current device (for callers sizing work);
 * returns TWELL_ERR_CUDA without a device. */
TWELL_API twell_status twell_device_info(int32_t* sm_count, int32_t* cc_major, int32_t* cc_minor);

#ifdef __cplusplus
}
#endif

#endif /* TWELL_GB300_H */
