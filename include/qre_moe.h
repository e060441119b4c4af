/*
 * qre_moe.h -- C ABI of the GB300 routed-expert MoE library.
 *
 * One MoE layer's routed experts, resident in HBM as compact per-layer banks,
 * evaluated for decode tokens by hand-written sm_103a kernels.  The layer
 * computes (FreeToken PR #732, "apply the weight scales of nvfp4 gguf
 * tensors", section "Design"):
 *
 *     h = x @ W_gate_up^T;   g = h_gate * s_gate,  u = h_up * s_up
 *     y = (silu(g) * u  @ W_down^T) * s_down * routing_weight,  summed over routes
 *
 * with the per-expert scale bank [E,4] fp32 = (s_gate, s_up, s_down, 1), and
 * the pipeline of FreeToken PR #704 ("serve GGUF experts on the cpu and hybrid
 * backends through ggml-cpu", section "How it plugs into the CPU executor"):
 * prep_input (bf16 hidden -> q8_1, or kept float for BF16 rows), gate_up (a dot
 * over every gate and up row of the routed expert, then the activation),
 * prep_inter (intermediate -> the down type's input), down (a dot over every
 * output row per route) and the sum over routes.
 *
 * Conventions for every call below:
 *   - Return value: MOE_OK (0) or a negative moe_status.  No call throws, and
 *     no call aborts the process.
 *   - "device pointer" means memory of the current CUDA device; "stream" is a
 *     cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - moe_decode and the test hooks are asynchronous on the given stream; they
 *     allocate nothing, never synchronize, and may be captured into a CUDA
 *     graph.  Kernels are launched with programmatic dependent launch, so
 *     consecutive layers overlap their prologues.
 *   - The caller owns x, ids, weights, out and the workspace.  The library
 *     owns each bank (unless created with MOE_SRC_DEVICE_BORROW).
 */
#ifndef QRE_MOE_H
#define QRE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bank row types.  Row layouts (row = K values, rows stored back to back):
 *   MOE_BF16 : K little-endian bf16 (2K bytes).  FreeToken issue #194, "avoid
 *              max-stride padding ...", Proposed design: BF16 rows run through
 *              a float kernel, not the block-quantized one.
 *   MOE_Q8_0 : K/32 blocks of {fp16 d; int8 q[32]} (34 bytes), value d*q.
 *   MOE_Q4_K : K/256 super-blocks of 144 bytes {fp16 d; fp16 dmin;
 *              uint8 scales[12] (8 packed 6-bit (sc, m) pairs); uint8 qs[128]},
 *              value d*sc_j*q - dmin*m_j (GGUF Q4_K bit layout).
 *   MOE_NVFP4: K/2 code bytes (E2M1; element 2i in the low nibble of byte i)
 *              then K/16 UE4M3 scale bytes, one per 16 values (Strata PR #292,
 *              "NVFP4 routed experts ...", Summary/Pipeline: group 16).  The
 *              per-expert weight_scale_2 lives in the scale bank, not the row.
 *   MOE_Q6_K : K/256 super-blocks of 210 bytes {uint8 ql[128]; uint8 qh[64];
 *              int8 scales[16]; fp16 d}; value v = 128n + 32c + l of a
 *              super-block has the low nibble c/2 of ql[64n + 32(c mod 2) + l]
 *              and bits 2c, 2c+1 of qh[32n + l] as its 6-bit code q, and the
 *              value d*scales[v/16]*(q - 32) (GGUF Q6_K bit layout; one of the
 *              ggml weight types FreeToken PR #704 lists, "How it plugs into
 *              the CPU executor").
 *   MOE_Q4_0 : K/32 blocks of {fp16 d; uint8 qs[16]} (18 bytes); value j < 16
 *              is the low nibble of qs[j], value j+16 its high nibble, value
 *              d*(q - 8) (GGUF Q4_0 bit layout; the CPU format of FreeToken
 *              PR #704, "Tests").
 *   MOE_Q4_1 : K/32 blocks of {fp16 d; fp16 m; uint8 qs[16]} (20 bytes), codes
 *              as MOE_Q4_0, value d*q + m.
 *   MOE_Q5_0 : K/32 blocks of {fp16 d; uint8 qh[4]; uint8 qs[16]} (22 bytes):
 *              the low 4 code bits as MOE_Q4_0, bit j of the little-endian
 *              word qh is the fifth bit of value j; value d*(q - 16).
 *   MOE_Q5_1 : K/32 blocks of {fp16 d; fp16 m; uint8 qh[4]; uint8 qs[16]}
 *              (24 bytes), codes as MOE_Q5_0, value d*q + m.
 *   MOE_Q5_K : K/256 super-blocks of 176 bytes {fp16 d; fp16 dmin; uint8
 *              scales[12]; uint8 qh[32]; uint8 qs[128]}: scales and the low 4
 *              code bits as MOE_Q4_K, bit j of qh[l] the fifth bit of value l
 *              of sub-block j; value d*sc_j*q - dmin*m_j.
 *   MOE_MXFP4: K/32 blocks of {uint8 e; uint8 qs[16]} (17 bytes), E2M1 codes
 *              laid out as MOE_Q4_0, value E2M1(code) * 2^(e - 127); e = 255
 *              (not a finite E8M0 scale) must not occur.
 *   MOE_F16  : K little-endian IEEE fp16 (2K bytes).
 *   MOE_F32  : K little-endian IEEE fp32 (4K bytes).
 * (Q4_1 through MXFP4, F16 and F32 are the remaining types of FreeToken PR
 * #704's synthetic list, "Validation"; GGUF bit layouts.)  Float rows (BF16,
 * F16, F32) take the activations unquantized, as BF16 does: x as its bf16
 * values, the intermediate as fp32; a float gate_up or down may sit beside a
 * quantized one of the other projection.  Banks must be readable
 * up to the next 16-byte boundary past their last row.
 * Gate_up and down may be of different types (e.g. Q4_K gate_up with Q6_K
 * down, the pairing of a Q4_K_M checkpoint). */
typedef enum {
  MOE_BF16 = 0, MOE_Q8_0 = 1, MOE_Q4_K = 2, MOE_NVFP4 = 3, MOE_Q6_K = 4, MOE_Q4_0 = 5,
  MOE_Q4_1 = 6, MOE_Q5_0 = 7, MOE_Q5_1 = 8, MOE_Q5_K = 9, MOE_MXFP4 = 10, MOE_F16 = 11, MOE_F32 = 12
} moe_type;

typedef enum {
  MOE_OK = 0,
  MOE_EINVAL = -1,        /* bad argument: null pointer, size, geometry, alignment */
  MOE_EUNSUPPORTED = -2,  /* valid but not built: e.g. a type or shape outside the limits */
  MOE_ENOMEM = -3,        /* device allocation failed (bank creation only) */
  MOE_ECUDA = -4,         /* a CUDA runtime call failed; see moe_last_cuda_error() */
  MOE_EDEVICE = -5        /* moe_get_error found a device-side error bit */
} moe_status;

/* Device-side error bits (sticky in the workspace, read by moe_get_error). */
enum {
  MOE_DEVERR_BAD_ID = 1,   /* a topk id outside [0, E): that route contributed zero */
  MOE_DEVERR_TIMEOUT = 2   /* a bounded wait on a TMA copy ran out; outputs are invalid */
};

/* Limits of this build. */
enum {
  MOE_MAX_E = 1024,        /* experts per layer */
  MOE_MAX_TOPK = 32,       /* routes per token */
  MOE_DECODE_T_CHUNK = 64, /* tokens per internal decode pass (larger T is split) */
  MOE_LINEAR_MAX_T = 8     /* tokens per moe_linear call */
};

/* The GLU of the layer, glu(g, u) = act(g) * u (FreeToken PR #732, "Design":
 * y = (glu(g, u) @ W_down^T) * s_down * routing_weight; its "Other checks"
 * run experts with gelu_tanh and silu):
 *   MOE_GLU_SILU      : act(g) = g / (1 + exp(-g))
 *   MOE_GLU_GELU_TANH : act(g) = g/2 * (1 + tanh(sqrt(2/pi) * (g + 0.044715 g^3)))
 * Both are evaluated in fp32. */
typedef enum { MOE_GLU_SILU = 0, MOE_GLU_GELU_TANH = 1 } moe_glu;

typedef struct {
  int32_t H;             /* hidden size; multiple of 256 for Q4_K gate_up, else of 32 */
  int32_t I;             /* intermediate size; multiple of 32 (256 for Q4_K down) */
  int32_t E;             /* experts, 1..MOE_MAX_E */
  int32_t top_k;         /* routes per token, 1..min(E, MOE_MAX_TOPK) */
  int32_t gate_up_type;  /* moe_type of the merged gate_up rows [E, 2I, H]: rows [0,I) gate, [I,2I) up */
  int32_t down_type;     /* moe_type of the down rows [E, H, I] */
  int32_t glu;           /* moe_glu: the activation of the gate half (0 = SiLU) */
} moe_layer_geom;

/* Where moe_bank_create reads the rows from. */
enum {
  MOE_SRC_HOST = 0,          /* host memory: copied to a library-owned device bank */
  MOE_SRC_DEVICE = 1,        /* device memory: copied (device to device) */
  MOE_SRC_DEVICE_BORROW = 2  /* device memory used in place: the caller keeps it alive and
                                unmodified until moe_bank_destroy; base 16-byte aligned and
                                readable up to the next 16-byte boundary past its end */
};

typedef struct moe_bank moe_bank;   /* opaque */

/* Bytes of one row of k values of `type` (FreeToken PR #704, "How it plugs
 * into the CPU executor": a bank holds rows of row_bytes(type, K)).
 * Returns 0 when k is not a whole number of the type's blocks. */
size_t moe_row_bytes(int32_t type, int64_t k);

/* Create a layer bank.  gate_up: E*2I rows of row_bytes(gate_up_type, H);
 * down: E*H rows of row_bytes(down_type, I); both compact at the exact row
 * stride (FreeToken issue #194, Proposed design: no padding to another layer's
 * stride).  gate_up_bytes / down_bytes must equal those products exactly.
 * scale_bank: [E,4] fp32 (s_gate, s_up, s_down, unused) in the same memory
 * kind as the rows (host for MOE_SRC_HOST, else device), or NULL for all
 * ones; it is always copied.  Synchronizes `stream` before returning.
 * Errors: MOE_EINVAL (geometry, sizes, null or misaligned pointer),
 * MOE_EUNSUPPORTED, MOE_ENOMEM, MOE_ECUDA.  *out is set only on success. */
int moe_bank_create(const moe_layer_geom* geom,
                    const void* gate_up, size_t gate_up_bytes,
                    const void* down, size_t down_bytes,
                    const float* scale_bank, int32_t src_kind,
                    void* stream, moe_bank** out);

/* Free a bank (waits for the device to finish with it).  NULL is a no-op. */
int moe_bank_destroy(moe_bank* bank);

/* Copy the bank's geometry to *out. */
int moe_bank_geometry(const moe_bank* bank, moe_layer_geom* out);

/* Fold a router's per-expert output scale into the bank's s_down column:
 * s_down[e] = fp32(s_down[e] * per_expert_scale[e]) for e < E (IEEE fp32
 * multiply), after which the router's weights are used without that scale
 * (FreeToken PR #732, "Design": the converter folds Gemma-4's per_expert_scale
 * into the down experts' scale).  per_expert_scale: E fp32 values in host
 * (src_kind MOE_SRC_HOST) or device (MOE_SRC_DEVICE) memory, 4-byte aligned.
 * Synchronizes `stream`; must not run concurrently with a decode on the bank.
 * Errors: MOE_EINVAL (null, src_kind, alignment), MOE_ENOMEM, MOE_ECUDA. */
int moe_bank_fold_down_scale(moe_bank* bank, const float* per_expert_scale, int32_t src_kind, void* stream);

/* Workspace bytes moe_decode needs for batches of up to max_tokens tokens
 * (0 on bad arguments).  The workspace holds the quantized activations, the
 * intermediate, per-block counters and the sticky error word. */
size_t moe_workspace_bytes(const moe_bank* bank, int32_t max_tokens);

/* Clear a freshly allocated workspace (error word and counters), async on
 * `stream`.  Call once after allocating; calls never leave it dirty. */
int moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Decode T tokens through one MoE layer.
 *   x:        device, bf16 [T, H] row-major.
 *   topk_ids: device, int32 [T, top_k]; an id outside [0, E) makes its route
 *             contribute zero and sets MOE_DEVERR_BAD_ID.
 *   topk_w:   device, fp32 [T, top_k] routing weights.
 *   out:      device, bf16 [T, H]; out[t] = bf16(sum over k in order k = 0..top_k-1
 *             of the route's fp32 result), with no atomics.
 *   ws:       device workspace of at least moe_workspace_bytes(bank, T') bytes
 *             for T' = min(T, MOE_DECODE_T_CHUNK), 256-byte aligned, initialised
 *             once by moe_workspace_init.  Calls sharing a workspace must be
 *             ordered on one stream.
 * T = 0 is a no-op.  Errors: MOE_EINVAL, MOE_ECUDA (launch failure). */
int moe_decode(const moe_bank* bank, const void* x, int32_t T,
               const int32_t* topk_ids, const float* topk_w, void* out,
               void* ws, size_t ws_bytes, void* stream);

/* moe_decode without a caller-provided workspace, for callers that cannot
 * allocate device memory: plugins whose host framework owns every device
 * allocation and hands the library only its own tensors, and latency-critical
 * serving paths where a cudaMalloc may synchronize the device.  The pages have
 * no counterpart to this entry point; it exists for those callers.
 *
 * The workspace is a fixed MOE_NOALLOC_WS_BYTES array in device memory that
 * every GPU loading this library holds until the process exits.  The first
 * call on a device (and the first after that device's context was torn down
 * and created again) looks up that array's device address with that device
 * current; make that first call before any stream capture.  Every call
 * shares the array and starts by clearing its error word; the array keeps the
 * last call's contents otherwise.  Calls that overlap on the GPU (on different
 * streams, or from different threads) race on it, so order them.  This call
 * itself reports no device-side error bits: a bad id contributes zero, and a
 * bounded wait that ran out leaves the outputs invalid; read the bits with
 * moe_get_error(NULL, 0, stream, &bits), which reads this array's error word.
 * Arguments as for moe_decode.  Returns MOE_EINVAL, without launching
 * anything, when one pass of this call would need more workspace than
 * MOE_NOALLOC_WS_BYTES (moe_workspace_bytes(bank, T) tells), and never calls
 * cudaMalloc or cudaFree. */
enum { MOE_NOALLOC_WS_BYTES = 4 << 20 };
int moe_decode_noalloc(const moe_bank* bank, const void* x, int32_t T,
                       const int32_t* topk_ids, const float* topk_w, void* out,
                       void* stream);

/* ---------------------------------------------------------------- prompt path
 * Grouped expert GEMMs for a prompt chunk (Strata PR #292, "Summary/Pipeline":
 * the prompt path, W4A8 with q8_1 activations, W4A4 with activations
 * quantized to NVFP4 on the fly, or FP16 with activations kept in fp16).
 * NVFP4 gate_up and down banks only, H and I multiples of 256; other banks
 * return MOE_EUNSUPPORTED. */
enum { MOE_PREFILL_W4A4 = 0, MOE_PREFILL_W4A8 = 1, MOE_PREFILL_FP16 = 2, MOE_PREFILL_W4A4_FIXED = 3 };

/* Workspace bytes moe_prefill_grouped needs for T tokens in `mode`; 0 if the
 * bank or mode is unsupported or T < 1. */
size_t moe_prefill_workspace_bytes(const moe_bank* bank, int32_t T, int32_t mode);

/* Prompt-path layer: out[t] = bf16(sum over k of the routed expert's output
 * times s_down * topk_w[t, k]), the same layer as moe_decode with the prompt
 * path's activation quantization.  Steps: routes sorted by expert (stable);
 * x quantized per token (W4A4: per 16 values a UE4M3 scale = amax/6 and E2M1
 * codes, both rounded to nearest even with saturation, global scale 1; W4A8:
 * the q8_1 rule of the decode path; FP16: x rounded to fp16, nearest even);
 * a grouped gate_up GEMM on the tensor cores over the exactly dequantized
 * operands (fp32 accumulation of exact products) with s_gate, s_up and the
 * GLU in an fp32 epilogue that requantizes the intermediate the same way as x
 * (FP16: rounds it to fp16); a grouped down GEMM whose epilogue scales by
 * s_down * routing weight; the route sum in fp32, rounded once to bf16.
 * W4A8, FP16 and MOE_PREFILL_W4A4_FIXED (W4A4 arithmetic, the same
 * kernels up to the down epilogue) add k = 0..K-1 in order, so repeated
 * calls give identical bits.  MOE_PREFILL_W4A4 on the block-scaled FP4
 * tensor cores adds each route into its token's fp32 sum as the down tiles
 * finish (bulk reductions at L2, no per-route fp32 rows in HBM), so the order
 * of those K additions, and with it the last fp32 bits of a sum, can differ
 * between calls (the error bound is the same for every order).  On a bank
 * without the FP4 tensor-core layout both W4A4 modes take the fixed order.
 * x: bf16 [T, H] (device, 16-byte aligned); topk_ids int32 and topk_w fp32
 * [T, K] (device); out bf16 [T, H] (device, 8-byte aligned); ws: device,
 * 256-byte aligned, >= moe_prefill_workspace_bytes(bank, T, mode) bytes (no
 * initialization needed; each call starts by clearing its error word).
 * Asynchronous on `stream`; a route whose id is outside [0, E) contributes
 * zero and sets MOE_DEVERR_BAD_ID (read with moe_get_error on the same
 * workspace). */
int moe_prefill_grouped(const moe_bank* bank, const void* x, int32_t T,
                        const int32_t* topk_ids, const float* topk_w, int32_t mode,
                        void* out, void* ws, size_t ws_bytes, void* stream);

/* Number of kernels one moe_decode call of T tokens launches on this bank
 * (for graph builders and launch accounting), or a negative status. */
int moe_decode_kernel_count(const moe_bank* bank, int32_t T);

/* Device staging bytes moe_decode_host needs for T tokens (0 on bad arguments). */
size_t moe_decode_io_bytes(const moe_bank* bank, int32_t T);

/* Byte offsets of topk_ids, topk_w and out in the staging layout of
 * moe_decode_host for T tokens (x is at offset 0): offsets[0..2].  Returns
 * MOE_EINVAL on bad arguments. */
int moe_decode_io_offsets(const moe_bank* bank, int32_t T, size_t* offsets);

/* moe_decode on host buffers: copies x (bf16 [T, H]), topk_ids (int32 [T, K])
 * and topk_w (fp32 [T, K]) from the host into `io` (device, 256-byte aligned,
 * >= moe_decode_io_bytes(bank, T) bytes), decodes, and copies the bf16
 * [T, H] result back to `out` on the host, all asynchronous on `stream`
 * (host buffers must be pinned for the copies to overlap and to be
 * capturable in a CUDA graph; the result is in `out` once the stream has
 * reached this point).  When topk_ids and topk_w sit at x plus the offsets
 * of moe_decode_io_offsets, the three inputs move in one copy.  Workspace as
 * for moe_decode. */
int moe_decode_host(const moe_bank* bank, const void* x, int32_t T,
                    const int32_t* topk_ids, const float* topk_w, void* out,
                    void* io, size_t io_bytes, void* ws, size_t ws_bytes, void* stream);

/* Read and clear the workspace's sticky device error bits (synchronizes
 * `stream`).  *dev_err receives the MOE_DEVERR_* bits; returns MOE_EDEVICE if
 * any was set, MOE_OK otherwise.  ws = NULL (ws_bytes ignored) reads the
 * fixed workspace of moe_decode_noalloc on the current device; this too
 * allocates nothing. */
int moe_get_error(void* ws, size_t ws_bytes, void* stream, int32_t* dev_err);

/* Text for a moe_status value (static storage). */
const char* moe_status_string(int status);

/* The last CUDA error text seen by the library on this thread (static storage). */
const char* moe_last_cuda_error(void);

/* ---------------------------------------------------------------- test hooks
 * Not on the decode path; they run the same device functions the decode
 * kernels use, so parity tests can check intermediate results bit for bit. */

/* Quantize n fp32 values (device, n a multiple of 32) to q8_1 blocks of 36
 * bytes {fp16 d; fp16 s; int8 q[32]} (device, n/32 blocks): d = amax/127,
 * q = round-half-even(x/d) (0 when d = 0), s = d * sum(q), all in fp32 with
 * d and s stored as fp16 -- the input quantizer of the decode path. */
int moe_quantize_q8_1(const float* x, int64_t n, void* out_blocks, void* stream);

/* Integer block dot products of quantized rows (device, nrows rows of
 * row_bytes(type, k)) against q8_1 activation blocks (device, k/32 blocks of
 * 36 bytes).  out: device int32 [nrows, nb] with nb = k/16 for MOE_NVFP4 (one
 * per 16-value block, sum of (2*E2M1 code value) * q), k/32 for MOE_Q8_0 and
 * MOE_Q4_K (sum of code * q; Q4_K per 32-value sub-block), k/16 for MOE_Q6_K
 * (sum of (code - 32) * q per 16-value scale group), k/32 for MOE_Q4_0 (sum of
 * (code - 8) * q), MOE_Q5_0 (sum of (code - 16) * q), MOE_Q4_1, MOE_Q5_1 and
 * MOE_Q5_K (sum of code * q) and MOE_MXFP4 (sum of (2*E2M1 code value) * q).
 * Float types (MOE_BF16, MOE_F16, MOE_F32) are MOE_EINVAL. */
int moe_debug_block_dots(int32_t type, const void* rows, int32_t nrows, int32_t k,
                         const void* act_blocks, int32_t* out, void* stream);

/* Run moe_decode, then export workspace stages (any pointer may be NULL):
 *   x_blocks:     the q8_1 blocks of x, [T, H/32] x 36 bytes (quantized gate_up only);
 *   inter:        the fp32 intermediate silu(g)*u, [T*top_k, I];
 *   inter_blocks: its q8_1 blocks, [T*top_k, I/32] x 36 bytes (quantized down only).
 * Requires T <= MOE_DECODE_T_CHUNK.  Routes with a bad id leave their rows
 * unspecified. */
int moe_debug_decode_stages(const moe_bank* bank, const void* x, int32_t T,
                            const int32_t* topk_ids, const float* topk_w, void* out,
                            void* ws, size_t ws_bytes, void* stream,
                            void* x_blocks, float* inter, void* inter_blocks);

/* Run moe_prefill_grouped, then export its stages (any pointer may be NULL):
 *   xq:   the quantized x, W4A4: [T] rows of H/2 E2M1 code bytes (element 2i
 *         in the low nibble of byte i) then H/16 UE4M3 scale bytes; W4A8:
 *         [T, H/32] q8_1 blocks of 36 bytes {fp16 d; fp16 s; int8 q[32]};
 *   off:  int32 [E+1], the first sorted row of each expert (off[E] = valid routes);
 *   perm: int32 [T*K], the route index t*K+k of each sorted row;
 *   i16:  fp16 [T*K, I], the dequantized requantized intermediate of each
 *         sorted row. */
int moe_debug_prefill_stages(const moe_bank* bank, const void* x, int32_t T,
                             const int32_t* topk_ids, const float* topk_w, int32_t mode,
                             void* out, void* ws, size_t ws_bytes, void* stream,
                             void* xq, int32_t* off, int32_t* perm, void* i16);

/* Dense quantized linear with a per-output-row scale in its epilogue:
 *   out[t, n] = bf16(row_scale[n] * sum_k W[n, k] * q8_1(x[t])[k])
 * for t < T, n < N (FreeToken PR #732, "Design": a dense linear multiplies
 * its matmul result by its scale; a fused module of several tensors, e.g.
 * qkv or gate_up, carries ggml_scale, one fp32 value per output row, each
 * part's scale or 1).  x is quantized to q8_1 per 32 values inside the call
 * (the decode path's prep_input), each 32-value block's integer dot is exact,
 * the block scales and row_scale are applied in fp32, and the output is
 * rounded once to bf16 (ties to even).
 *   type:      any quantized moe_type (float types are MOE_EUNSUPPORTED); an
 *              NVFP4 tensor's weight_scale_2 goes into row_scale
 *   rows:      device, N rows of moe_row_bytes(type, K) bytes back to back,
 *              16-byte aligned and readable up to the next 16-byte boundary
 *              past the last row
 *   row_scale: device fp32 [N], or NULL for ones
 *   x:         device bf16 [T][K], 16-byte aligned; out: device bf16 [T][N]
 *   T:         1..MOE_LINEAR_MAX_T; T = 0 is a no-op
 *   dev_err:   device uint32 or NULL; OR-ed with MOE_DEVERR_TIMEOUT if a
 *              bounded wait ran out
 * Asynchronous on `stream`; allocates nothing.  Errors: MOE_EINVAL (null
 * pointer, alignment, sizes), MOE_EUNSUPPORTED (type, or T*K too large for
 * the activations to stay in shared memory: about 150 K values), MOE_ECUDA. */
int moe_linear(int32_t type, const void* rows, int32_t N, int32_t K, const float* row_scale,
               const void* x, int32_t T, void* out, uint32_t* dev_err, void* stream);

/* ---------------------------------------------------------------- expert cache
 * For expert banks larger than the GPU's memory (FreeToken issue #194,
 * "avoid max-stride padding for heterogeneous GGUF expert banks", Proposed
 * design): a byte budget is split into exact-geometry slot pools, one per
 * tuple of row sizes, each with its own LRU state keyed by (layer, expert);
 * missed experts are copied from the layer's compact rows straight into
 * their slots.  A pool is a bank whose experts are its slots, so a request
 * decodes with moe_decode on moe_cache_bank() after its routing ids are
 * replaced by the slot ids moe_cache_acquire returns. */

/* Slots per geometry for a byte budget: with w_g = selections[g] (routed
 * expert selections per token of the layers of geometry g, e.g. layers x
 * top_k), n_g = floor(budget * w_g / sum_h w_h * expert_bytes[h]); the bytes
 * left over then go one slot at a time to the smallest expert size that still
 * fits.  (For 39 Q4_K layers of 5.0625 MiB experts and 8 BF16 layers of
 * 18 MiB experts at top-10, the budget of 480 x 18 MiB gives 988 + 202 slots,
 * the pages' Controlled A/B.)  slots: int64 [ngeom] out.  Host only. */
int moe_cache_plan(int64_t budget_bytes, int32_t ngeom, const int64_t* expert_bytes,
                   const int64_t* selections, int64_t* slots);

/* The LRU state of one pool, on the host (no device memory). */
typedef struct moe_slot_table moe_slot_table;
int moe_slot_table_create(int32_t nslots, moe_slot_table** out);
int moe_slot_table_destroy(moe_slot_table* table);

/* Slots for one request of layer `layer`: ids int32 [n] (host) are expert ids
 * of that layer; ids outside [0, E) get slot -1.  The request's distinct
 * valid experts that are resident (hits) become the most recent first; each
 * missing one then takes the least recently used slot (never-used slots are
 * the least recent, lowest index first) and becomes the most recent, so a
 * request never evicts its own experts.  Writes slot_ids [n], and for each
 * miss, in first-occurrence order, fill_slots[i] / fill_experts[i] (capacity:
 * the number of slots) with *nfill the count.  MOE_EUNSUPPORTED if the request
 * names more distinct experts than there are slots (nothing changes). */
int moe_slot_table_acquire(moe_slot_table* table, int32_t layer, const int32_t* ids, int32_t n, int32_t E,
                           int32_t* slot_ids, int32_t* fill_slots, int32_t* fill_experts, int32_t* nfill);
int moe_slot_table_stats(const moe_slot_table* table, int64_t* hits, int64_t* misses);

/* One exact-geometry pool of nslots slots on the device (1..MOE_MAX_E; the
 * geometry's E is ignored, its top_k must not exceed nslots).  Allocates
 * nslots expert rows of each projection (+256 bytes) and zeroes them on
 * `stream`. */
typedef struct moe_cache moe_cache;
int moe_cache_create(const moe_layer_geom* geom, int32_t nslots, void* stream, moe_cache** out);
int moe_cache_destroy(moe_cache* cache);

/* The pool as a bank (owned by the cache): decode with slot ids. */
moe_bank* moe_cache_bank(moe_cache* cache);

/* Make one request's experts resident: moe_slot_table_acquire on the pool's
 * LRU state, then for each miss three copies on `stream` (cudaMemcpyAsync,
 * any memory the device can address; pinned host memory keeps them
 * asynchronous): the expert's 2I gate_up rows and H down rows from the
 * layer's compact banks (gate_up [E][2I][row bytes], down [E][H][row bytes],
 * the same layout moe_bank_create takes) and its scale row from scales [E][4]
 * (NULL: ones).  Decode on the same stream after this call; the sources must
 * stay valid until the copies complete.  *nfill (may be NULL) = misses.  If
 * enqueueing a copy fails (MOE_ECUDA), the slots this request assigned are
 * untagged, so a later request copies those experts again. */
int moe_cache_acquire(moe_cache* cache, int32_t layer, const void* gate_up, const void* down,
                      const float* scales, int32_t E, const int32_t* ids, int32_t n, int32_t* slot_ids,
                      int32_t* nfill, void* stream);

/* Cumulative hits and misses (distinct experts per request) and bytes copied. */
int moe_cache_stats(const moe_cache* cache, int64_t* hits, int64_t* misses, int64_t* copied_bytes);

/* Forget which expert every slot holds (LRU order and counters unchanged):
 * the next request for each expert misses and copies it again.  Host only. */
int moe_slot_table_invalidate(moe_slot_table* table);
int moe_cache_invalidate(moe_cache* cache);

/* A byte-denominated bank arena (FreeToken issue #194, Proposed design):
 * pools carved from one caller-owned device buffer at disjoint offsets.
 * moe_cache_bytes: the device bytes of a pool of nslots slots (gate_up rows,
 * then down rows, each region 256-byte aligned with 256 bytes of slack); 0
 * on bad arguments.  moe_cache_create_at: moe_cache_create on
 * [base, base + moe_cache_bytes) of caller memory (base 256-byte aligned,
 * bytes >= moe_cache_bytes; MOE_EINVAL otherwise), zeroed on `stream`; the
 * memory is not freed by moe_cache_destroy. */
size_t moe_cache_bytes(const moe_layer_geom* geom, int32_t nslots);
int moe_cache_create_at(const moe_layer_geom* geom, int32_t nslots, void* base, size_t bytes, void* stream,
                        moe_cache** out);

/* Full-layer prefill overlay (FreeToken issue #194, Proposed design: prefill
 * of a whole layer runs on one shared overlay of the arena, and the geometry
 * pools are invalidated before the overlay is written).  An overlay holds one
 * layer's complete bank -- all E experts' gate_up rows, then its down rows,
 * at the layer's exact stride -- at `base`, which may overlap pools of the
 * same arena; size the arena region for the largest layer that will use it.
 * moe_overlay_bytes: bytes an overlay of this geometry needs (0 on bad
 * arguments).  moe_overlay_create: base 256-byte aligned, bytes >=
 * moe_overlay_bytes (MOE_EINVAL otherwise); allocates only the bank's scale
 * rows.  moe_overlay_bank: the overlay as a bank for moe_prefill_grouped (or
 * moe_decode), owned by the overlay. */
typedef struct moe_overlay moe_overlay;
size_t moe_overlay_bytes(const moe_layer_geom* geom);
int moe_overlay_create(const moe_layer_geom* geom, void* base, size_t bytes, void* stream, moe_overlay** out);
int moe_overlay_destroy(moe_overlay* overlay);
moe_bank* moe_overlay_bank(moe_overlay* overlay);

/* Write one layer into the overlay: first, on the host, every pool of
 * pools[0..npools) whose rows share any byte with the overlay is invalidated
 * (moe_cache_invalidate); then the layer's compact rows (gate_up
 * [E][2I][row bytes], down [E][H][row bytes], any memory the device can
 * address; device-addressable sources are copied by one kernel) and its
 * scale rows (scales [E][4], NULL: ones) are copied in on `stream`.  Run the
 * prefill on the same stream.  A later fill of an overlapping pool
 * overwrites the overlay: load it again before the next prefill. */
int moe_overlay_load(moe_overlay* overlay, moe_cache* const* pools, int32_t npools, const void* gate_up,
                     const void* down, const float* scales, void* stream);

/* Tensor-core check: D[128, N] = A[128, K] * B[N, K]^T with fp16 A and B
 * (device, row-major), fp32 D (device, row-major), computed with the tcgen05
 * kind::f16 MMA on swizzled shared-memory tiles that the prompt-path GEMMs
 * use.  K a positive multiple of 64, N a multiple of 16 in [16, 256], A and B
 * 16-byte aligned.  *dev_err (device int32, caller-zeroed) gets bit 0 if a
 * bounded wait for the MMA ran out. */
int moe_debug_tc_gemm(const void* A, const void* B, int32_t K, int32_t N, float* D,
                      int32_t* dev_err, void* stream);

/* Block-scaled FP4 tensor-core check: D[128, N] = sum over k of
 * (E2M1(A[m][k]) * UE4M3(sA[m][k/16])) * (E2M1(B[n][k]) * UE4M3(sB[n][k/16]))
 * on the tcgen05 kind::mxf4nvf4 MMA (per-16 UE4M3 scales in tensor memory)
 * that the W4A4 prompt path runs on (Strata PR #292, "Summary/Pipeline":
 * W4A4 on FP4 MMA).  A: device, 128 rows of K/2 bytes of E2M1 codes (value
 * 2i in the low nibble of byte i); B: N rows likewise; sA, sB: 128 / N rows
 * of K/16 UE4M3 bytes; D: device fp32 [128][N].  K a positive multiple of
 * 256, N a multiple of 16 in [16, 256] (above 128 the scales of B take eight
 * tensor-memory columns a MMA), A, B, sA, sB 16-byte aligned.
 * *dev_err (device int32, caller-zeroed) gets bit 0 if a bounded wait for
 * the MMA ran out. */
int moe_debug_fp4_gemm(const void* A, const void* scale_A, const void* B, const void* scale_B, int32_t K,
                       int32_t N, float* D, int32_t* dev_err, void* stream);

/* Failure-detection check (the auxiliary failure detection of the build, not
 * an operation of the pages): one thread runs one of the kernels' bounded
 * waits on an mbarrier whose phase nothing completes, so the wait runs out
 * and the kernel sets MOE_DEVERR_TIMEOUT in *dev_err and returns; the
 * context stays usable.
 *   mode 0: the sleeping-poll wait of the decode kernels, `limit` polls of at
 *           most about 0.5 ms each;
 *   mode 1: the spinning wait of the grouped and prompt-path kernels, `limit`
 *           microseconds of device time.
 *   limit:  1 .. MOE_DEBUG_WAIT_MAX.
 *   dev_err: device uint32 (caller-zeroed); OR-ed with MOE_DEVERR_TIMEOUT.
 * Asynchronous on `stream`; allocates nothing.  Errors: MOE_EINVAL. */
enum { MOE_DEBUG_WAIT_MAX = 64 };
int moe_debug_wait_timeout(int32_t mode, int32_t limit, uint32_t* dev_err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QRE_MOE_H */
