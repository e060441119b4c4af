// Internal declarations shared by the C-ABI layer and the kernels.
#pragma once
#include <cuda.h>   // CUtensorMap (the type only; the library links the runtime alone)
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

struct moe_bank;   // the C ABI's opaque bank (api.cu)

namespace qre {

constexpr int kMaxE = 1024;
constexpr int kSortBlocks = 32;   // blocks of the prompt path's two-pass route sort
constexpr int kMaxTopK = 32;
constexpr int kTChunk = 64;
constexpr int kMaxGridCtas = 256;   // CTAs of the fused kernel's grid barrier

// Everything one decode pass (at most kTChunk tokens) needs, by value in
// kernel parameter space.
struct DecodeParams {
  int H, I, E, K, T;
  int glu;                 // kGluSilu or kGluGeluTanh
  int gu_type, dn_type;
  int rb_gu, rb_dn;
  const uint8_t* gu_bank;  // [E][2I][rb_gu]
  const uint8_t* dn_bank;  // [E][H][rb_dn]
  const float* scales;     // [E][4]
  const uint16_t* x;       // bf16 [T][H]
  const int32_t* ids;      // [T][K]
  const float* w;          // [T][K]
  uint16_t* out;           // bf16 [T][H]
  // workspace
  uint32_t* err;
  int8_t* xq; float* xd; int* xsum; uint16_t* xsh;   // q8_1 of x: [T][H], [T][H/32]
  float* inter;                                         // [T*K][I]
  int8_t* iq; float* id; int* isum; uint16_t* ish;   // q8_1 of inter: [T*K][I], [T*K][I/32]
  unsigned* cnt;                                        // [min(E, T*K)][I/32]
  int cnt_len;
  // launch shape
  int g_gu, g_dn;          // grid sizes
  int ps;                  // gate_up pairs per stage
  int gu_up_off;           // byte offset of the up rows inside a gate_up stage buffer
  int gu_stage_bytes, gu_nstage;
  int dn_rows_max;         // max rows per down CTA
  int dn_rs;               // rows per down stage piece
  int dn_slots_per_stage;
  int dn_piece_bytes;      // bytes reserved per (slot, row piece) inside a down stage
  int dn_stage_bytes, dn_nstage;
  int w0;                  // gate_up cost model: cost per pair = w0 + tokens of the expert
  int gu_act_smem, gu_act_bytes;  // stage x's activations in shared memory (bytes reserved)
  int dn_act_smem, dn_act_bytes;  // stage the intermediate's activations in shared memory
  int maxnt;               // routes per register-held work item: 1 (small batches) or 4
  // fused small-batch layer kernel (layer_small.cu)
  int use_ls;              // 1: one k_layer_small launch replaces k_gate_up + k_down
  int g_ls;                // its grid (one CTA per SM)
  int ls_ns, ls_sb;        // ring depth and bytes per ring slot
  unsigned* bar;           // grid-barrier words in the workspace (epoch, then two arrival counts, 128 B apart)
};

// The prompt path (prefill.cu): routes sorted by expert, then two grouped
// GEMMs on the tensor cores (gate_up, down) and a fixed-order combine.
enum PfMode : int { PF_W4A4 = 0, PF_W4A8 = 1, PF_FP16 = 2 };
struct PfParams {
  int H, I, E, K, T, RT;
  int glu;
  int mode;
  int rb_gu, rb_dn;
  const uint8_t* gu_bank;   // NVFP4 rows [E][2I][rb_gu]
  const uint8_t* dn_bank;   // NVFP4 rows [E][H][rb_dn]
  const float* scales;      // [E][4]
  const uint16_t* x;        // bf16 [T][H]
  const int32_t* ids;       // [T][K]
  const float* w;           // [T][K]
  uint16_t* out;            // bf16 [T][H]
  // workspace
  uint32_t* err;
  int* off;                 // [E+1] first sorted row of each expert; off[E] = valid routes
  int* perm;                // [RT]  route index of each sorted row
  int* bcnt;                // [kSortBlocks][E] the sort's per-block expert counts
  int* inv;                 // [RT]  W4A4 on the FP4 tensor cores: sorted row of each route (-1: invalid id), else null
  uint8_t* xs;              // [RT][H/2 + H/16] W4A4 on the FP4 tensor cores: NVFP4 x by sorted row, else null
  float* ysum;              // [T][H] fp32 token sums that k_pf_quant zeroes (FP4 tensor cores, completion-order sum), else null
  uint8_t* xq;              // quantized x: NVFP4 rows [T][H/2 + H/16] (W4A4) or q8_1 blocks [T][H/32][36] (W4A8)
  uint16_t* x16;            // fp16 [T][H]: the dequantized quantized x (the gate_up A operand)
  uint16_t* x16lo;          // fp16 [T][H], W4A8 only: q*d - x16 (x16 + x16lo carries q*d to ~2^-22)
  uint16_t* i16;            // fp16 [RT][I]: the dequantized requantized intermediate, sorted rows
  float* y;                 // fp32 [RT][H]: down output of each route times s_down * w, by route index
                            // (W4A4 on the FP4 tensor cores: fp32 [T][H] token sums, zeroed by k_pf_quant)
};

// The W4A4 prompt path on the block-scaled FP4 tensor cores (prefill.cu):
// x quantized to NVFP4 per token and written to every sorted row of its
// routes (k_pf_quant), then two grouped GEMMs (tcgen05 kind::mxf4nvf4, both operands
// fed by 2-D TMA, per-16 UE4M3 scales in tensor memory); the down GEMM adds
// each route's scaled row into its token's fp32 sum by bulk reductions at L2,
// and one pass rounds the sums to bf16.  NVFP4 rows are codes (K/2 bytes)
// then scales (K/16 bytes).
struct Pf4Params {
  CUtensorMap map_xs, map_xss;    // xs [RT][H/2 + H/16]: code boxes 128 B x 128 rows (swizzled), scale boxes 16 x 128
  CUtensorMap map_wgu, map_wgus;  // gate_up bank [E*2I][H/2 + H/16], the same boxes
  CUtensorMap map_in, map_ins;    // in4 [RT][I/2 + I/16]
  CUtensorMap map_wdn, map_wdns;  // down bank [E*H][I/2 + I/16]
  int H, I, E, K, T, RT;
  int glu;
  int export_i16;                 // also write the dequantized intermediate as fp16 (inspection)
  const float* scales;            // [E][4]
  const int32_t* ids;             // [T][K]
  const float* w;                 // [T][K]
  uint32_t* err;
  const int* off;                 // [E+1]
  const int* perm;                // [RT]
  uint8_t* xs;                    // NVFP4 x by sorted row [RT][H/2 + H/16]
  uint8_t* in4;                   // NVFP4 intermediate by sorted row [RT][I/2 + I/16]
  uint16_t* i16;                  // fp16 [RT][I] (export_i16 only)
  float* y;                       // fp32 [T][H]: each token's sum of its routes' scaled down outputs
                                  // (fixed: fp32 [RT][H], each route's scaled down output by route index)
  uint16_t* out;                  // bf16 [T][H]
  int fixed;                      // route sum in the order k = 0..K-1 (k_pf4_combine) instead of L2 reductions
};

// The dense path (decode_tc.cu): BF16 gate_up and down banks at batches the
// fused kernel cannot hold.  Routes sorted by expert, the routed tokens'
// hidden states gathered in that order, then two grouped GEMMs on the tensor
// cores (weights streamed by 2-D TMA into swizzled tiles) and a fixed-order
// route sum.  H and I are multiples of 64.
struct DtParams {
  CUtensorMap map_gu;       // gate_up bank as bf16 [E*2I][H], box 64 x 128 rows, 128-byte swizzle
  CUtensorMap map_dn;       // down bank as bf16 [E*H][I], box 64 x 128 rows
  CUtensorMap map_xs;       // xs: bf16 [RTp][H], box 64 x 16 rows
  CUtensorMap map_ih;       // ih: bf16 [2*RTp][I] (hi rows, then lo rows), box 64 x 16 rows
  int H, I, E, K, T, RT, RTp;
  int glu;
  const float* scales;      // [E][4]
  const uint16_t* x;        // bf16 [T][H]
  const int32_t* ids;       // [T][K]
  const float* w;           // [T][K]
  uint16_t* out;            // bf16 [T][H]
  // workspace
  uint32_t* err;
  int* off;                 // [E+1] first sorted row of each expert; off[E] = valid routes
  int* perm;                // [RTp] route index of each sorted row
  uint16_t* xs;             // bf16 [RTp][H]: x of the token of each sorted row
  uint16_t* ih;             // bf16 [2*RTp][I]: intermediate of each sorted row as hi + lo (a = hi + lo to ~2^-16)
  float* inter;             // fp32 [RT][I]: the intermediate by route index (as the other paths leave it)
  float* y;                 // fp32 [RT][H]: down output of each route times s_down * w, by route index
};

// The batched path for Q4_K and NVFP4 banks (decode_qb.cu) at batches the
// fused kernel cannot hold: each token's x quantized to q8_1 once, then two
// grouped CUDA-core kernels (each sorts the routes by expert itself) that stream one 256-value
// K chunk of 256 weight rows per 2-D TMA stage (144 bytes a row in both
// formats) and dot each decoded block with up to kQbTileTokens routed tokens
// (tiles handed out heaviest expert first), and the fixed-order route sum.
// A q8_1 block record is 8 bytes: the fp16-rounded scale as fp32, then the
// int32 code sum.  H and I are multiples of 256.
constexpr int kQbTileTokens = 8;    // routed tokens per tile of the batched kernels
struct QbParams {
  // banks as byte matrices [E*2I][rb_gu] and [E*H][rb_dn], boxes of 128 rows:
  // Q4_K, Q4_0: map_w* boxes 144 bytes wide (256 values); NVFP4: map_w* boxes
  // the 128 code bytes of a chunk (128-byte swizzle), map_w*s its 16 scale bytes
  CUtensorMap map_wgu, map_wdn, map_wgus, map_wdns;
  CUtensorMap map_xq;       // xq [T][H], box 256 x 1 row
  CUtensorMap map_xr;       // xrec [T][H/4], box 64 x 1 row
  CUtensorMap map_iq;       // iqs [RTp][I], box 256 x kQbTileTokens rows
  CUtensorMap map_is;       // iss [RTp][I/4], box 64 x kQbTileTokens rows
  int wt;                   // W_Q4_K, W_Q4_0 or W_NVFP4 (both projections)
  int H, I, E, K, T, RT, RTp;
  int glu;
  const float* scales;      // [E][4]
  const uint16_t* x;        // bf16 [T][H]
  const int32_t* ids;       // [T][K]
  const float* w;           // [T][K]
  uint16_t* out;            // bf16 [T][H]
  // workspace
  uint32_t* err;
  unsigned* sched;          // [0], [1]: next tile of gate_up / down
  uint8_t* xrec;            // q8_1 block records of x [T][H/32][8]
  int8_t* iqs;              // q8_1 codes of the intermediate for each sorted row [RTp][I]
  uint8_t* iss;             // block records [RTp][I/32][8]
  // per-token / per-route planes, also left for inspection
  int8_t* xq; float* xd; int* xsum; uint16_t* xsh;
  float* inter;
  int8_t* iq; float* id; int* isum; uint16_t* ish;
  float* y;                 // fp32 [RT][H]: down output of each route times s_down * w, by route index
};

// Sizes of the dynamic shared memory of each kernel for these params.
size_t gate_up_smem_bytes(const DecodeParams& p);
size_t down_smem_bytes(const DecodeParams& p);

// Launches (all with programmatic dependent launch on `stream`).
cudaError_t launch_prep(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_gate_up(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_down(const DecodeParams& p, cudaStream_t stream);

// Fused small-batch layer kernel.
size_t layer_small_smem_bytes(const DecodeParams& p);
bool layer_small_fits(const DecodeParams& p);
cudaError_t launch_layer_small(const DecodeParams& p, cudaStream_t stream);

// Dense path for BF16 banks (four launches: route + gather, gate_up, down, route sum).
constexpr int kDtLaunches = 4;
cudaError_t launch_dense(const DtParams& p, cudaStream_t stream);

// Batched path for Q4_K banks (four launches: route + quantize, gate_up + requantize, down, route sum).
constexpr int kQbLaunches = 4;
cudaError_t launch_qbatch(const QbParams& p, cudaStream_t stream);

// Test hooks.
cudaError_t launch_quantize_q8_1_blocks(const float* x, int64_t n, uint8_t* out, cudaStream_t stream);
cudaError_t launch_block_dots(int type, const uint8_t* rows, int nrows, int k, const uint8_t* act,
                              int32_t* out, cudaStream_t stream);
struct Pf4Params;
cudaError_t launch_prefill(const PfParams& p, cudaStream_t stream, const Pf4Params* fp4 = nullptr);
// The W4A4 GEMMs on FP4 (after k_pf_sort and k_pf_quant of launch_prefill).
cudaError_t launch_prefill_fp4(const Pf4Params& q, cudaStream_t stream);
cudaError_t launch_tc_gemm_check(const uint16_t* A, const uint16_t* B, int K, int N, float* D, int* err,
                                 cudaStream_t stream);
cudaError_t launch_wait_timeout(int mode, uint32_t limit, uint32_t* err, cudaStream_t stream);
cudaError_t launch_fp4_gemm_check(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, int K,
                                  int N, float* D, int* err, cudaStream_t stream);
cudaError_t launch_export_q8(const int8_t* q, const float* d, const uint16_t* s, int64_t nblocks,
                             uint8_t* out, cudaStream_t stream);

// Dense quantized linear with per-output-row scales (linear.cu).
constexpr int kLinearMaxT = 8;
struct LinParams {
  int type;                 // WType of the rows (a quantized type)
  int N, K, T, rb;          // rows, values per row, tokens, bytes per row
  const uint8_t* rows;      // [N][rb]
  const float* row_scale;   // [N] or null (ones)
  const uint16_t* x;        // bf16 [T][K]
  uint16_t* out;            // bf16 [T][N]
  uint32_t* err;            // error word (kErrTimeout) or null
  int rps, stage_bytes, nstage, act_bytes, grid;   // launch plan (plan_linear)
};
bool plan_linear(LinParams& p);
size_t linear_smem_bytes(const LinParams& p);
cudaError_t launch_linear(const LinParams& p, cudaStream_t stream);

// Bank internals the expert cache (cache.cu) writes: the device scale rows
// [E][4]; and the library's CUDA error report (sets moe_last_cuda_error).
float* bank_scales(moe_bank* b);
int report_cuda_error(cudaError_t e, const char* what);

int sm_count();

}  // namespace qre
