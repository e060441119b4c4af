// C ABI of the routed-expert MoE library (declared in include/qre_moe.h):
// bank residency, workspace layout, argument checks and kernel dispatch.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/qre_moe.h"
#include "formats.cuh"
#include "internal.h"

using namespace qre;

struct moe_bank {
  moe_layer_geom geom;
  int rb_gu, rb_dn;
  uint8_t* gu;      // [E][2I][rb_gu] (+ slack)
  uint8_t* dn;      // [E][H][rb_dn]  (+ slack)
  float* scales;    // [E][4]
  bool owns_rows;
  int device;
  // Grouped path for batches the fused kernel cannot hold: kGroupedDense
  // (BF16 gate_up and down, H and I multiples of 64) or kGroupedQuant (Q4_K
  // or NVFP4 gate_up and down, H and I multiples of 256), with the bank's
  // rows as 2-D tensors for TMA.
  int grouped;
  CUtensorMap map_gu;       // dense: bf16 [E*2I][H], box 64 x 128; Q4_K: bytes [E*2I][rb_gu], box 144 x 128;
                            // NVFP4: the same bytes, box 128 x 128 (code bytes, 128-byte swizzle)
  CUtensorMap map_dn;       // the same for [E*H] down rows
  CUtensorMap map_gus;      // NVFP4: the same bytes, box 16 x 128 (scale bytes)
  CUtensorMap map_dns;
};

namespace {

thread_local char g_cuda_err[256] = "no error";

int cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", what, cudaGetErrorString(e));
  return MOE_ECUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// cuTensorMapEncodeTiled, looked up once through the runtime (the library
// does not link the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && f)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// A row-major bf16 matrix [rows][cols] as a 2-D tensor map: boxes of 64
// columns (128 bytes) x box_rows rows, written to shared memory with the
// 128-byte swizzle; reads outside the matrix fill zeros.
bool map_bf16_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major byte matrix [rows][cols] as a 2-D tensor map: boxes of
// box_cols bytes (a multiple of 16) x box_rows rows, copied to shared memory
// densely (rows box_cols bytes apart), or with the 128-byte swizzle (box_cols
// = 128); reads outside the matrix fill zeros.
bool map_byte_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                   uint32_t box_rows, bool swizzle128 = false) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

enum { kGroupedNone = 0, kGroupedDense = 1, kGroupedQuant = 2 };

int grouped_kind(const moe_layer_geom& g) {
  if (g.gate_up_type == MOE_BF16 && g.down_type == MOE_BF16 && g.H % 64 == 0 && g.I % 64 == 0) return kGroupedDense;
  if ((g.gate_up_type == MOE_Q4_K || g.gate_up_type == MOE_Q4_0 || g.gate_up_type == MOE_NVFP4) &&
      g.down_type == g.gate_up_type &&
      g.H % 256 == 0 && g.I % 256 == 0)
    return kGroupedQuant;
  return kGroupedNone;
}

int geom_check(const moe_layer_geom* g) {
  if (!g) return MOE_EINVAL;
  if (g->E < 1 || g->E > kMaxE || g->top_k < 1 || g->top_k > kMaxTopK || g->top_k > g->E) return MOE_EINVAL;
  if (g->H < 32 || g->I < 32 || g->H > (1 << 16) || g->I > (1 << 16)) return MOE_EINVAL;
  if (g->gate_up_type < MOE_BF16 || g->gate_up_type > MOE_F32) return MOE_EINVAL;
  if (g->down_type < MOE_BF16 || g->down_type > MOE_F32) return MOE_EINVAL;
  if (row_bytes_of(g->gate_up_type, g->H) == 0 || row_bytes_of(g->down_type, g->I) == 0) return MOE_EINVAL;
  if (g->H % 32 != 0 || g->I % 32 != 0) return MOE_EINVAL;
  if (g->glu != MOE_GLU_SILU && g->glu != MOE_GLU_GELU_TANH) return MOE_EINVAL;
  return MOE_OK;
}

// Rows of the bank that one down CTA owns, and the tokens of one decode pass.
struct Shape {
  int g_gu, g_dn, rows_max, t_chunk;
};

Shape decode_shape(const moe_layer_geom& g) {
  Shape s;
  // sized for one CTA per SM (the most rows per down CTA); batches of up to
  // two tokens run two CTAs per SM (make_params)
  s.g_gu = sm_count();
  s.g_dn = sm_count();
  if (s.g_dn > g.H) s.g_dn = g.H;
  s.rows_max = (g.H + s.g_dn - 1) / s.g_dn;
  // keep the per-route down results (T*K*rows_max fp32) within 96 KiB of shared memory
  int t = (96 * 1024) / (4 * g.top_k * s.rows_max);
  if (t > kTChunk) t = kTChunk;
  if (t < 1) t = 1;
  s.t_chunk = t;
  return s;
}

struct WsLayout {
  size_t err, bar, xq, xd, xsum, xsh, inter, iq, id, isum, ish, cnt, total;
  int cnt_len;
  size_t d_y;                              // grouped paths: per-route down output
  size_t d_off, d_perm, d_xs, d_ih;        // dense path: routes sorted by expert, gathered x, intermediate hi + lo
  size_t q_sched, q_xr, q_iq, q_is;        // batched path: tile counters, x block records, sorted intermediate
  int RTp;
};

WsLayout ws_layout(const moe_layer_geom& g, int T) {
  WsLayout L;
  const size_t A = 256;
  const size_t RT = (size_t)T * g.top_k;
  size_t o = 0;
  L.err = o; o = align_up(o + 4, A);
  L.bar = o; o = align_up(o + 128 * 3, A);   // the fused kernel's barrier: epoch, then two arrival counts
  L.xq = o; o = align_up(o + (size_t)T * g.H, A);
  L.xd = o; o = align_up(o + 4 * (size_t)T * (g.H / 32), A);
  L.xsum = o; o = align_up(o + 4 * (size_t)T * (g.H / 32), A);
  L.xsh = o; o = align_up(o + 2 * (size_t)T * (g.H / 32), A);
  L.inter = o; o = align_up(o + 4 * RT * g.I, A);
  L.iq = o; o = align_up(o + RT * g.I, A);
  L.id = o; o = align_up(o + 4 * RT * (g.I / 32), A);
  L.isum = o; o = align_up(o + 4 * RT * (g.I / 32), A);
  L.ish = o; o = align_up(o + 2 * RT * (g.I / 32), A);
  const size_t S = (size_t)g.E < RT ? (size_t)g.E : RT;
  L.cnt_len = (int)(S * (g.I / 32));
  L.cnt = o; o = align_up(o + 4 * (size_t)L.cnt_len, A);
  L.RTp = (int)((RT + 31) / 32 * 32);
  L.d_off = L.d_perm = L.d_y = L.d_xs = L.d_ih = L.q_sched = L.q_xr = L.q_iq = L.q_is = 0;
  const int gk = grouped_kind(g);
  if (gk != kGroupedNone) {
    L.d_y = o; o = align_up(o + 4 * RT * g.H, A);
  }
  if (gk == kGroupedDense) {
    L.d_off = o; o = align_up(o + 4 * ((size_t)g.E + 1), A);
    L.d_perm = o; o = align_up(o + 4 * (size_t)L.RTp, A);
    L.d_xs = o; o = align_up(o + 2 * (size_t)L.RTp * g.H, A);
    L.d_ih = o; o = align_up(o + 2 * 2 * (size_t)L.RTp * g.I, A);
  } else if (gk == kGroupedQuant) {
    L.q_sched = o; o = align_up(o + 4 * 4, A);
    L.q_xr = o; o = align_up(o + (size_t)T * (g.H / 4), A);
    L.q_iq = o; o = align_up(o + (size_t)L.RTp * g.I, A);
    L.q_is = o; o = align_up(o + (size_t)L.RTp * (g.I / 4), A);
  }
  L.total = o;
  return L;
}

// Shape of the fused small-batch kernel: one CTA per SM, a ring of ~32 KiB
// slots shared by gate_up and down stages, activations in shared memory.
// Leaves p.use_ls = 0 when it does not fit (the two-kernel path then runs).
void plan_layer_small(const moe_layer_geom& g, int T, DecodeParams& p) {
  DecodeParams q = p;
  q.g_ls = sm_count();
  if (q.g_ls > g.H) q.g_ls = g.H;
  if (q.g_ls > kMaxGridCtas) return;
  const int rows_max = (g.H + q.g_ls - 1) / q.g_ls;
  q.dn_rows_max = rows_max;
  int rs = (24 * 1024) / q.rb_dn;
  rs = rs < 1 ? 1 : (rs > rows_max ? rows_max : rs);
  q.dn_rs = rs;
  q.dn_piece_bytes = (int)align_up((size_t)rs * q.rb_dn + 16, 128);
  int sps = (32 * 1024) / q.dn_piece_bytes;
  q.dn_slots_per_stage = sps < 1 ? 1 : (sps > 16 ? 16 : sps);
  int ps = (32 * 1024) / (2 * q.rb_gu);
  ps = ps < 1 ? 1 : (ps > 32 ? 32 : ps);
  q.ps = ps;
  q.gu_up_off = (int)align_up((size_t)ps * q.rb_gu + 16, 128);
  const int gu_stage = 2 * q.gu_up_off, dn_stage = q.dn_slots_per_stage * q.dn_piece_bytes;
  q.ls_sb = gu_stage > dn_stage ? gu_stage : dn_stage;
  const size_t RT = (size_t)T * g.top_k;
  const size_t xa = is_float_w(g.gate_up_type) ? 2 * (size_t)T * g.H : (size_t)T * g.H + 8 * (size_t)T * (g.H / 32);
  q.gu_act_smem = 1;
  q.gu_act_bytes = (int)align_up(xa, 16);
  if (is_float_w(g.down_type)) {
    const size_t ia = 4 * RT * g.I;
    q.dn_act_smem = ia <= 48 * 1024 ? 1 : 0;
    q.dn_act_bytes = q.dn_act_smem ? (int)align_up(ia, 16) : 0;
  } else {
    q.dn_act_smem = 1;
    q.dn_act_bytes = (int)align_up(RT * g.I + 8 * RT * (g.I / 32), 16);
  }
  q.ls_ns = 0;
  const size_t fixed = layer_small_smem_bytes(q);
  const size_t budget = 210 * 1024;
  if (fixed + 2 * (size_t)(q.ls_sb + 16) > budget) return;
  int ns = (int)((budget - fixed) / (q.ls_sb + 16));
  q.ls_ns = ns > 8 ? 8 : ns;
  q.use_ls = 1;
  if (!layer_small_fits(q)) return;
  p = q;
}

DecodeParams make_params(const moe_bank* b, const WsLayout& L, uint8_t* ws, const Shape& sh, int T) {
  const moe_layer_geom& g = b->geom;
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.H = g.H; p.I = g.I; p.E = g.E; p.K = g.top_k; p.T = T;
  p.gu_type = g.gate_up_type; p.dn_type = g.down_type;
  p.glu = g.glu;
  p.rb_gu = b->rb_gu; p.rb_dn = b->rb_dn;
  p.gu_bank = b->gu; p.dn_bank = b->dn; p.scales = b->scales;
  p.err = reinterpret_cast<uint32_t*>(ws + L.err);
  p.bar = reinterpret_cast<unsigned*>(ws + L.bar);
  p.xq = reinterpret_cast<int8_t*>(ws + L.xq);
  p.xd = reinterpret_cast<float*>(ws + L.xd);
  p.xsum = reinterpret_cast<int*>(ws + L.xsum);
  p.xsh = reinterpret_cast<uint16_t*>(ws + L.xsh);
  p.inter = reinterpret_cast<float*>(ws + L.inter);
  p.iq = reinterpret_cast<int8_t*>(ws + L.iq);
  p.id = reinterpret_cast<float*>(ws + L.id);
  p.isum = reinterpret_cast<int*>(ws + L.isum);
  p.ish = reinterpret_cast<uint16_t*>(ws + L.ish);
  p.cnt = reinterpret_cast<unsigned*>(ws + L.cnt);
  p.cnt_len = L.cnt_len;
  // Batches of up to two tokens take the two-kernel path (x quantized inside
  // k_gate_up, the intermediate requantized inside k_down) when the
  // activations fit in shared memory; larger batches take k_prep + k_gate_up
  // + k_down.
  {
    const size_t RT0 = (size_t)T * g.top_k;
    const size_t gu_need = is_float_w(g.gate_up_type) ? 2 * (size_t)T * g.H : (size_t)T * g.H * 5 / 4;
    const size_t dn_need = is_float_w(g.down_type) ? 0 : RT0 * g.I * 5 / 4;
    p.maxnt = (T <= 2 && gu_need <= 48 * 1024 && dn_need <= 64 * 1024) ? 1 : 4;
  }
  p.g_gu = sh.g_gu;
  p.g_dn = sh.g_dn;
  if (p.g_dn > g.H) p.g_dn = g.H;
  const int rows_max = (g.H + p.g_dn - 1) / p.g_dn;
  // gate_up stages: ~32 KiB of (gate, up) row pairs, ~96 KiB in flight
  int ps = (32 * 1024) / (2 * p.rb_gu);
  if (ps < 1) ps = 1;
  if (ps > 32) ps = 32;
  p.ps = ps;
  p.gu_up_off = (int)align_up((size_t)ps * p.rb_gu + 16, 128);
  p.gu_stage_bytes = 2 * p.gu_up_off;
  int ns = (96 * 1024) / p.gu_stage_bytes;
  p.gu_nstage = ns < 2 ? 2 : (ns > 8 ? 8 : ns);
  // down stages: pieces of <= 24 KiB rows of one expert, grouped to ~32 KiB
  p.dn_rows_max = rows_max;
  int rs = (24 * 1024) / p.rb_dn;
  if (rs < 1) rs = 1;
  if (rs > rows_max) rs = rows_max;
  p.dn_rs = rs;
  p.dn_piece_bytes = (int)align_up((size_t)rs * p.rb_dn + 16, 128);
  int sps = (32 * 1024) / p.dn_piece_bytes;
  p.dn_slots_per_stage = sps < 1 ? 1 : (sps > 16 ? 16 : sps);
  p.dn_stage_bytes = p.dn_slots_per_stage * p.dn_piece_bytes;
  int dns = (64 * 1024) / p.dn_stage_bytes;
  p.dn_nstage = dns < 2 ? 2 : (dns > 8 ? 8 : dns);
  // activations staged in shared memory when they fit (always on the two-kernel path)
  const size_t RT = (size_t)T * g.top_k;
  const size_t gu_act = is_float_w(g.gate_up_type) ? 2 * (size_t)T * g.H
                                                     : (size_t)T * g.H + 8 * (size_t)T * (g.H / 32);
  p.gu_act_smem = (p.maxnt == 1 || gu_act <= 24 * 1024) ? 1 : 0;
  p.gu_act_bytes = p.gu_act_smem ? (int)align_up(gu_act, 16) : 0;
  const size_t dn_act = is_float_w(g.down_type) ? 4 * RT * g.I : RT * g.I + 8 * RT * (g.I / 32);
  p.dn_act_smem = ((p.maxnt == 1 && !is_float_w(g.down_type)) || dn_act <= 24 * 1024) ? 1 : 0;
  p.dn_act_bytes = p.dn_act_smem ? (int)align_up(dn_act, 16) : 0;
  // ring depths: no deeper than the stages a CTA is expected to have, and
  // small enough at low token counts for a down CTA to sit beside a gate_up CTA
  const size_t U = (size_t)g.E < RT ? (size_t)g.E : RT;
  const size_t pairs = (U * g.I + p.g_gu - 1) / p.g_gu;
  int gst = (int)((pairs + ps - 1) / ps) + 2;
  p.gu_nstage = gst < 2 ? 2 : (gst < p.gu_nstage ? gst : p.gu_nstage);
  const int dpieces = (rows_max + rs - 1) / rs;
  int dst = dpieces * (int)((U + p.dn_slots_per_stage - 1) / p.dn_slots_per_stage);
  p.dn_nstage = dst < 2 ? 2 : (dst < p.dn_nstage ? dst : p.dn_nstage);
  plan_layer_small(g, T, p);
  // The grouped paths take over from the fused kernel once they are faster
  // (measured: BF16 from 2 tokens; Q4_K from 20 routes per pass, the
  // Laguna-shaped layer at T=2; NVFP4 between 16 and 32 routes, the
  // Qwen3-30B-A3B-shaped layer at T=2 and T=4; Q4_0 takes the Q4_K
  // threshold: the same bytes per 256 values and the same kernel).
  const int RTn = T * g.top_k;
  if ((b->grouped == kGroupedDense && T >= 2) || (b->grouped == kGroupedQuant && RTn >= 20)) p.use_ls = 0;
  switch (p.gu_type) {
    case W_NVFP4: p.w0 = 2; break;
    case W_Q4_K: p.w0 = 3; break;
    case W_Q8_0: p.w0 = 2; break;
    case W_Q6_K: p.w0 = 3; break;
    case W_Q5_K: p.w0 = 3; break;
    case W_Q4_0: case W_Q4_1: case W_Q5_0: case W_Q5_1: case W_MXFP4: p.w0 = 2; break;
    default: p.w0 = 4; break;
  }
  return p;
}

}  // namespace

namespace qre {   // internals the expert cache (cache.cu) uses
float* bank_scales(moe_bank* b) { return b ? b->scales : nullptr; }
int report_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
}  // namespace qre

extern "C" {

size_t moe_row_bytes(int32_t type, int64_t k) {
  if (k <= 0 || k > (1 << 30)) return 0;
  return (size_t)row_bytes_of(type, (int)k);
}

const char* moe_status_string(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument";
    case MOE_EUNSUPPORTED: return "unsupported";
    case MOE_ENOMEM: return "out of device memory";
    case MOE_ECUDA: return "CUDA error";
    case MOE_EDEVICE: return "device-side error flag set";
  }
  return "unknown status";
}

const char* moe_last_cuda_error(void) { return g_cuda_err; }

int moe_bank_create(const moe_layer_geom* geom, const void* gate_up, size_t gate_up_bytes, const void* down,
                    size_t down_bytes, const float* scale_bank, int32_t src_kind, void* stream, moe_bank** out) {
  if (!out || !gate_up || !down) return MOE_EINVAL;
  int st = geom_check(geom);
  if (st) return st;
  if (src_kind < MOE_SRC_HOST || src_kind > MOE_SRC_DEVICE_BORROW) return MOE_EINVAL;
  const moe_layer_geom& g = *geom;
  const int rb_gu = row_bytes_of(g.gate_up_type, g.H), rb_dn = row_bytes_of(g.down_type, g.I);
  const size_t want_gu = (size_t)g.E * 2 * g.I * rb_gu, want_dn = (size_t)g.E * g.H * rb_dn;
  if (gate_up_bytes != want_gu || down_bytes != want_dn) return MOE_EINVAL;
  if (src_kind == MOE_SRC_DEVICE_BORROW && (!aligned(gate_up, 16) || !aligned(down, 16))) return MOE_EINVAL;
  if (scale_bank && !aligned(scale_bank, 4)) return MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  moe_bank* b = new (std::nothrow) moe_bank;
  if (!b) return MOE_ENOMEM;
  std::memset(b, 0, sizeof(*b));
  b->geom = g;
  b->rb_gu = rb_gu;
  b->rb_dn = rb_dn;
  cudaGetDevice(&b->device);
  cudaError_t e;
  if (src_kind == MOE_SRC_DEVICE_BORROW) {
    b->gu = const_cast<uint8_t*>(static_cast<const uint8_t*>(gate_up));
    b->dn = const_cast<uint8_t*>(static_cast<const uint8_t*>(down));
    b->owns_rows = false;
  } else {
    b->owns_rows = true;
    if ((e = cudaMalloc(&b->gu, want_gu + 256)) != cudaSuccess) { delete b; cudaGetLastError(); return MOE_ENOMEM; }
    if ((e = cudaMalloc(&b->dn, want_dn + 256)) != cudaSuccess) {
      cudaFree(b->gu); delete b; cudaGetLastError(); return MOE_ENOMEM;
    }
    const cudaMemcpyKind kind = (src_kind == MOE_SRC_HOST) ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    if ((e = cudaMemcpyAsync(b->gu, gate_up, want_gu, kind, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(b->dn, down, want_dn, kind, s)) != cudaSuccess) {
      cudaFree(b->gu); cudaFree(b->dn); delete b; return cuda_fail(e, "bank copy");
    }
  }
  if ((e = cudaMalloc(&b->scales, 16 * (size_t)g.E)) != cudaSuccess) {
    if (b->owns_rows) { cudaFree(b->gu); cudaFree(b->dn); }
    delete b; cudaGetLastError(); return MOE_ENOMEM;
  }
  if (scale_bank) {
    const cudaMemcpyKind kind = (src_kind == MOE_SRC_HOST) ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    e = cudaMemcpyAsync(b->scales, scale_bank, 16 * (size_t)g.E, kind, s);
  } else {
    std::vector<float> ones(4 * (size_t)g.E, 1.0f);
    e = cudaMemcpyAsync(b->scales, ones.data(), 16 * (size_t)g.E, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    if (b->owns_rows) { cudaFree(b->gu); cudaFree(b->dn); }
    cudaFree(b->scales); delete b; return cuda_fail(e, "bank create");
  }
  // the grouped paths stream the rows with 2-D TMA: one tensor map per projection
  b->grouped = kGroupedNone;
  const int gk = grouped_kind(g);
  if (gk == kGroupedDense &&
      map_bf16_rows(&b->map_gu, b->gu, (uint64_t)g.E * 2 * g.I, (uint64_t)g.H, 128) &&
      map_bf16_rows(&b->map_dn, b->dn, (uint64_t)g.E * g.H, (uint64_t)g.I, 128))
    b->grouped = kGroupedDense;
  if (gk == kGroupedQuant && (g.gate_up_type == MOE_Q4_K || g.gate_up_type == MOE_Q4_0) &&
      map_byte_rows(&b->map_gu, b->gu, (uint64_t)g.E * 2 * g.I, (uint64_t)rb_gu, 144, 128) &&
      map_byte_rows(&b->map_dn, b->dn, (uint64_t)g.E * g.H, (uint64_t)rb_dn, 144, 128))
    b->grouped = kGroupedQuant;
  if (gk == kGroupedQuant && g.gate_up_type == MOE_NVFP4 &&
      map_byte_rows(&b->map_gu, b->gu, (uint64_t)g.E * 2 * g.I, (uint64_t)rb_gu, 128, 128, true) &&
      map_byte_rows(&b->map_dn, b->dn, (uint64_t)g.E * g.H, (uint64_t)rb_dn, 128, 128, true) &&
      map_byte_rows(&b->map_gus, b->gu, (uint64_t)g.E * 2 * g.I, (uint64_t)rb_gu, 16, 128) &&
      map_byte_rows(&b->map_dns, b->dn, (uint64_t)g.E * g.H, (uint64_t)rb_dn, 16, 128))
    b->grouped = kGroupedQuant;
  *out = b;
  return MOE_OK;
}

int moe_bank_destroy(moe_bank* b) {
  if (!b) return MOE_OK;
  cudaDeviceSynchronize();
  if (b->owns_rows) { cudaFree(b->gu); cudaFree(b->dn); }
  cudaFree(b->scales);
  delete b;
  return MOE_OK;
}

int moe_bank_geometry(const moe_bank* b, moe_layer_geom* out) {
  if (!b || !out) return MOE_EINVAL;
  *out = b->geom;
  return MOE_OK;
}

namespace {
__global__ void k_fold_down_scale(float* scales, const float* pes, int E) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < E) scales[4 * e + 2] = __fmul_rn(scales[4 * e + 2], pes[e]);
}
}  // namespace

int moe_bank_fold_down_scale(moe_bank* b, const float* per_expert_scale, int32_t src_kind, void* stream) {
  if (!b || !per_expert_scale) return MOE_EINVAL;
  if (src_kind != MOE_SRC_HOST && src_kind != MOE_SRC_DEVICE) return MOE_EINVAL;
  if (!aligned(per_expert_scale, 4)) return MOE_EINVAL;
  const int E = b->geom.E;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* tmp = nullptr;
  cudaError_t e = cudaMalloc(&tmp, sizeof(float) * (size_t)E);
  if (e != cudaSuccess) { cudaGetLastError(); return MOE_ENOMEM; }
  const cudaMemcpyKind kind = (src_kind == MOE_SRC_HOST) ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
  e = cudaMemcpyAsync(tmp, per_expert_scale, sizeof(float) * (size_t)E, kind, s);
  if (e == cudaSuccess) {
    k_fold_down_scale<<<(E + 255) / 256, 256, 0, s>>>(b->scales, tmp, E);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  cudaFree(tmp);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "fold_down_scale");
}

size_t moe_workspace_bytes(const moe_bank* b, int32_t max_tokens) {
  if (!b || max_tokens < 1) return 0;
  const Shape sh = decode_shape(b->geom);
  const int t = max_tokens < sh.t_chunk ? max_tokens : sh.t_chunk;
  return ws_layout(b->geom, t).total;
}

int moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < 256 || !aligned(ws, 256)) return MOE_EINVAL;
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "workspace init");
}

// Parameters of the dense path for one pass: the bank's tensor maps, two
// maps over this pass's workspace buffers, and the buffers themselves.
static bool dense_params(const moe_bank* b, const WsLayout& L, uint8_t* ws, const DecodeParams& p, DtParams& d) {
  const moe_layer_geom& g = b->geom;
  std::memset(&d, 0, sizeof(d));
  d.map_gu = b->map_gu;
  d.map_dn = b->map_dn;
  d.H = g.H; d.I = g.I; d.E = g.E; d.K = g.top_k; d.T = p.T;
  d.RT = p.T * g.top_k;
  d.RTp = L.RTp;
  d.glu = g.glu;
  d.scales = b->scales;
  d.x = p.x; d.ids = p.ids; d.w = p.w; d.out = p.out;
  d.err = p.err;
  d.off = reinterpret_cast<int*>(ws + L.d_off);
  d.perm = reinterpret_cast<int*>(ws + L.d_perm);
  d.xs = reinterpret_cast<uint16_t*>(ws + L.d_xs);
  d.ih = reinterpret_cast<uint16_t*>(ws + L.d_ih);
  d.inter = p.inter;
  d.y = reinterpret_cast<float*>(ws + L.d_y);
  if (!map_bf16_rows(&d.map_xs, d.xs, (uint64_t)L.RTp, (uint64_t)g.H, 16) ||
      !map_bf16_rows(&d.map_ih, d.ih, 2 * (uint64_t)L.RTp, (uint64_t)g.I, 16)) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "dense path: tensor map encode failed");
    return false;
  }
  return true;
}

// Parameters of the batched Q4_K path for one pass.
static bool qbatch_params(const moe_bank* b, const WsLayout& L, uint8_t* ws, const DecodeParams& p, QbParams& q) {
  const moe_layer_geom& g = b->geom;
  std::memset(&q, 0, sizeof(q));
  q.map_wgu = b->map_gu;
  q.map_wdn = b->map_dn;
  q.map_wgus = b->map_gus;
  q.map_wdns = b->map_dns;
  q.wt = g.gate_up_type;
  q.H = g.H; q.I = g.I; q.E = g.E; q.K = g.top_k; q.T = p.T;
  q.RT = p.T * g.top_k;
  q.RTp = L.RTp;
  q.glu = g.glu;
  q.scales = b->scales;
  q.x = p.x; q.ids = p.ids; q.w = p.w; q.out = p.out;
  q.err = p.err;
  q.sched = reinterpret_cast<unsigned*>(ws + L.q_sched);
  q.xrec = ws + L.q_xr;
  q.iqs = reinterpret_cast<int8_t*>(ws + L.q_iq);
  q.iss = ws + L.q_is;
  q.xq = p.xq; q.xd = p.xd; q.xsum = p.xsum; q.xsh = p.xsh;
  q.inter = p.inter;
  q.iq = p.iq; q.id = p.id; q.isum = p.isum; q.ish = p.ish;
  q.y = reinterpret_cast<float*>(ws + L.d_y);
  if (!map_byte_rows(&q.map_xq, q.xq, (uint64_t)p.T, (uint64_t)g.H, 256, 1) ||
      !map_byte_rows(&q.map_xr, q.xrec, (uint64_t)p.T, (uint64_t)g.H / 4, 64, 1) ||
      !map_byte_rows(&q.map_iq, q.iqs, (uint64_t)L.RTp, (uint64_t)g.I, 256, kQbTileTokens) ||
      !map_byte_rows(&q.map_is, q.iss, (uint64_t)L.RTp, (uint64_t)g.I / 4, 64, kQbTileTokens)) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "batched path: tensor map encode failed");
    return false;
  }
  return true;
}

static int decode_impl(const moe_bank* b, const void* x, int32_t T, const int32_t* ids, const float* w, void* out,
                       void* ws, size_t ws_bytes, void* stream, int* chunk_T) {
  if (!b || T < 0) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  if (!x || !ids || !w || !out || !ws) return MOE_EINVAL;
  if (!aligned(x, 16) || !aligned(out, 4) || !aligned(ids, 4) || !aligned(w, 4) || !aligned(ws, 256))
    return MOE_EINVAL;
  const moe_layer_geom& g = b->geom;
  const Shape sh = decode_shape(g);
  const int tc = T < sh.t_chunk ? T : sh.t_chunk;
  if (chunk_T) *chunk_T = tc;
  if (ws_bytes < ws_layout(g, tc).total) return MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int t0 = 0; t0 < T; t0 += tc) {
    const int tn = (T - t0) < tc ? (T - t0) : tc;
    const WsLayout L = ws_layout(g, tn);
    DecodeParams p = make_params(b, L, static_cast<uint8_t*>(ws), sh, tn);
    p.x = static_cast<const uint16_t*>(x) + (size_t)t0 * g.H;
    p.ids = ids + (size_t)t0 * g.top_k;
    p.w = w + (size_t)t0 * g.top_k;
    p.out = static_cast<uint16_t*>(out) + (size_t)t0 * g.H;
    cudaError_t e;
    if (p.use_ls) {
      if ((e = launch_layer_small(p, s)) != cudaSuccess) return cuda_fail(e, "layer launch");
      continue;
    }
    if (b->grouped == kGroupedDense) {
      DtParams d;
      if (!dense_params(b, L, static_cast<uint8_t*>(ws), p, d)) return MOE_ECUDA;
      if ((e = launch_dense(d, s)) != cudaSuccess) return cuda_fail(e, "dense launch");
      continue;
    }
    if (b->grouped == kGroupedQuant) {
      QbParams q;
      if (!qbatch_params(b, L, static_cast<uint8_t*>(ws), p, q)) return MOE_ECUDA;
      if ((e = launch_qbatch(q, s)) != cudaSuccess) return cuda_fail(e, "batched launch");
      continue;
    }
    if (p.maxnt != 1 && (e = launch_prep(p, s)) != cudaSuccess) return cuda_fail(e, "prep launch");
    if ((e = launch_gate_up(p, s)) != cudaSuccess) return cuda_fail(e, "gate_up launch");
    if ((e = launch_down(p, s)) != cudaSuccess) return cuda_fail(e, "down launch");
  }
  return MOE_OK;
}

int moe_decode(const moe_bank* b, const void* x, int32_t T, const int32_t* ids, const float* w, void* out, void* ws,
               size_t ws_bytes, void* stream) {
  return decode_impl(b, x, T, ids, w, out, ws, ws_bytes, stream, nullptr);
}

int moe_decode_kernel_count(const moe_bank* b, int32_t T) {
  if (!b || T < 0) return MOE_EINVAL;
  const moe_layer_geom& g = b->geom;
  const Shape sh = decode_shape(g);
  const int tc = T < sh.t_chunk ? T : sh.t_chunk;
  int n = 0;
  for (int t0 = 0; t0 < T; t0 += tc) {
    const int tn = (T - t0) < tc ? (T - t0) : tc;
    const WsLayout L = ws_layout(g, tn);
    const DecodeParams p = make_params(b, L, nullptr, sh, tn);
    n += p.use_ls                            ? 1
         : b->grouped == kGroupedDense       ? kDtLaunches
         : b->grouped == kGroupedQuant         ? kQbLaunches
         : (p.maxnt != 1 ? 3 : 2);
  }
  return n;
}

namespace {
struct IoLayout {
  size_t x, ids, w, out, total;
};
IoLayout io_layout(const moe_layer_geom& g, int T) {
  IoLayout L;
  size_t o = 0;
  L.x = o; o = align_up(o + 2 * (size_t)T * g.H, 256);
  L.ids = o; o = align_up(o + 4 * (size_t)T * g.top_k, 256);
  L.w = o; o = align_up(o + 4 * (size_t)T * g.top_k, 256);
  L.out = o; o = align_up(o + 2 * (size_t)T * g.H, 256);
  L.total = o;
  return L;
}
}  // namespace

size_t moe_decode_io_bytes(const moe_bank* b, int32_t T) {
  if (!b || T < 1) return 0;
  return io_layout(b->geom, T).total;
}

int moe_decode_io_offsets(const moe_bank* b, int32_t T, size_t* offsets) {
  if (!b || T < 1 || !offsets) return MOE_EINVAL;
  const IoLayout L = io_layout(b->geom, T);
  offsets[0] = L.ids;
  offsets[1] = L.w;
  offsets[2] = L.out;
  return MOE_OK;
}

int moe_decode_host(const moe_bank* b, const void* x, int32_t T, const int32_t* ids, const float* w, void* out,
                    void* io, size_t io_bytes, void* ws, size_t ws_bytes, void* stream) {
  if (!b || T < 0) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  if (!x || !ids || !w || !out || !io || !aligned(io, 256)) return MOE_EINVAL;
  const moe_layer_geom& g = b->geom;
  const IoLayout L = io_layout(g, T);
  if (io_bytes < L.total) return MOE_EINVAL;
  uint8_t* d = static_cast<uint8_t*>(io);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const uint8_t* hx = static_cast<const uint8_t*>(x);
  if (reinterpret_cast<const uint8_t*>(ids) == hx + L.ids && reinterpret_cast<const uint8_t*>(w) == hx + L.w) {
    // the host inputs already sit in the staging layout: one copy
    if ((e = cudaMemcpyAsync(d, x, L.w + 4 * (size_t)T * g.top_k, cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return cuda_fail(e, "decode_host: inputs to device");
  } else if ((e = cudaMemcpyAsync(d + L.x, x, 2 * (size_t)T * g.H, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
             (e = cudaMemcpyAsync(d + L.ids, ids, 4 * (size_t)T * g.top_k, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
             (e = cudaMemcpyAsync(d + L.w, w, 4 * (size_t)T * g.top_k, cudaMemcpyHostToDevice, s)) != cudaSuccess) {
    return cuda_fail(e, "decode_host: inputs to device");
  }
  const int st = decode_impl(b, d + L.x, T, reinterpret_cast<const int32_t*>(d + L.ids),
                             reinterpret_cast<const float*>(d + L.w), d + L.out, ws, ws_bytes, stream, nullptr);
  if (st) return st;
  if ((e = cudaMemcpyAsync(out, d + L.out, 2 * (size_t)T * g.H, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "decode_host: output to host");
  return MOE_OK;
}

// ------------------------------------------------------------------ decode without allocation
//
// The workspace of moe_decode_noalloc: a file-scope device array, so the call
// itself never allocates.  Host code cannot use `g_noalloc_ws` as a device
// address (on the host it names a stand-in); the device address is looked up
// once per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_ws[MOE_NOALLOC_WS_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
// Per device: the context the address was looked up in, and the address.
// Keyed on the context, so a device reset (a new context, the module loaded
// again) looks the address up again instead of using a stale one.
void* g_noalloc_ctx[kMaxDevices] = {};
void* g_noalloc_ptr[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && f)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

int noalloc_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return MOE_EUNSUPPORTED;
  const CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] && ctx && g_noalloc_ctx[dev] == (void*)ctx) {
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
  }
  // first call in this context: the lookup (which also makes the device's
  // context current if it was not yet)
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_ws);
  if (e != cudaSuccess || !ptr) return cuda_fail(e, "noalloc: cudaGetSymbolAddress");
  ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) ctx = nullptr;   // unknown: looked up again next call
  g_noalloc_ptr[dev] = ptr;
  g_noalloc_ctx[dev] = (void*)ctx;
  *out = ptr;
  return MOE_OK;
}
}  // namespace

int moe_decode_noalloc(const moe_bank* b, const void* x, int32_t T, const int32_t* ids, const float* w, void* out,
                       void* stream) {
  if (!b || T < 0) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  const Shape sh = decode_shape(b->geom);
  const int tc = T < sh.t_chunk ? T : sh.t_chunk;
  if (ws_layout(b->geom, tc).total > (size_t)MOE_NOALLOC_WS_BYTES) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err),
                  "moe_decode_noalloc: %zu workspace bytes needed, the static workspace holds %d",
                  ws_layout(b->geom, tc).total, (int)MOE_NOALLOC_WS_BYTES);
    return MOE_EINVAL;
  }
  void* ws = nullptr;
  int st = noalloc_workspace(&ws);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, s);   // the error word starts each call at zero
  if (e != cudaSuccess) return cuda_fail(e, "noalloc: clear error word");
  return decode_impl(b, x, T, ids, w, out, ws, (size_t)MOE_NOALLOC_WS_BYTES, stream, nullptr);
}

int moe_get_error(void* ws, size_t ws_bytes, void* stream, int32_t* dev_err) {
  if (!dev_err) return MOE_EINVAL;
  if (!ws) {   // the fixed workspace of moe_decode_noalloc
    const int st = noalloc_workspace(&ws);
    if (st) return st;
    ws_bytes = MOE_NOALLOC_WS_BYTES;
  }
  if (ws_bytes < 4) return MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && v) e = cudaMemsetAsync(ws, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "get_error");
  *dev_err = (int32_t)v;
  return v ? MOE_EDEVICE : MOE_OK;
}

int moe_quantize_q8_1(const float* x, int64_t n, void* out_blocks, void* stream) {
  if (!x || !out_blocks || n < 0 || n % 32 != 0 || !aligned(x, 4) || !aligned(out_blocks, 4)) return MOE_EINVAL;
  cudaError_t e = launch_quantize_q8_1_blocks(x, n, static_cast<uint8_t*>(out_blocks),
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "quantize_q8_1");
}

int moe_debug_block_dots(int32_t type, const void* rows, int32_t nrows, int32_t k, const void* act, int32_t* out,
                         void* stream) {
  if (!rows || !act || !out || nrows < 0 || k <= 0) return MOE_EINVAL;
  if (type <= MOE_BF16 || type > MOE_MXFP4) return MOE_EINVAL;   // quantized types only
  if (row_bytes_of(type, k) == 0 || !aligned(rows, 16) || !aligned(act, 4) || !aligned(out, 4)) return MOE_EINVAL;
  cudaError_t e = launch_block_dots(type, static_cast<const uint8_t*>(rows), nrows, k,
                                    static_cast<const uint8_t*>(act), out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "block_dots");
}

// ------------------------------------------------------------------ prompt path

namespace {

struct PfLayout {
  size_t err, off, perm, bcnt, inv, xq, x16, x16lo, i16, y, xs, in4, total;
};

// fp4: W4A4 on the FP4 tensor cores (the bank has its TMA maps): no fp16
// operands, and y holds one fp32 sum per token instead of one row per route
// unless the route sum takes the fixed order.
PfLayout pf_layout(const moe_layer_geom& g, int64_t T, int mode, bool fp4, bool fixed) {
  PfLayout L;
  const size_t A = 256;
  const size_t RT = (size_t)T * g.top_k;
  size_t o = 0;
  L.err = o; o = align_up(o + 4, A);
  L.off = o; o = align_up(o + 4 * ((size_t)g.E + 1), A);
  L.perm = o; o = align_up(o + 4 * RT, A);
  L.bcnt = o; o = align_up(o + 4 * (size_t)kSortBlocks * g.E, A);
  L.inv = o; o = align_up(o + (fp4 ? 4 * RT : 0), A);
  L.xq = o;
  o = align_up(o + (mode == PF_W4A4 ? (size_t)T * (g.H / 2 + g.H / 16)
                    : mode == PF_W4A8 ? (size_t)T * (g.H / 32) * 36 : 0), A);
  L.x16 = o; o = align_up(o + (fp4 ? 0 : 2 * (size_t)T * g.H), A);
  L.x16lo = o; o = align_up(o + (mode == PF_W4A8 ? 2 * (size_t)T * g.H : 0), A);
  L.i16 = o; o = align_up(o + 2 * RT * g.I, A);
  L.y = o; o = align_up(o + 4 * (fp4 && !fixed ? (size_t)T : RT) * g.H, A);
  // W4A4 on the FP4 tensor cores: NVFP4 rows of x and of the intermediate in sorted route order
  L.xs = L.in4 = 0;
  if (fp4) {
    L.xs = o; o = align_up(o + RT * (size_t)(g.H / 2 + g.H / 16), A);
    L.in4 = o; o = align_up(o + RT * (size_t)(g.I / 2 + g.I / 16), A);
  }
  L.total = o;
  return L;
}

bool pf_fp4(const moe_bank* b, int32_t mode) { return mode == PF_W4A4 && b->grouped == kGroupedQuant; }

// The public mode as the kernels' arithmetic mode and the route-sum order.
bool pf_mode(int32_t pub, int& mode, bool& fixed) {
  fixed = pub != MOE_PREFILL_W4A4;
  mode = pub == MOE_PREFILL_W4A4_FIXED ? PF_W4A4 : pub;
  return pub == MOE_PREFILL_W4A4 || pub == MOE_PREFILL_W4A8 || pub == MOE_PREFILL_FP16 ||
         pub == MOE_PREFILL_W4A4_FIXED;
}

int pf_check(const moe_bank* b, int32_t pub) {
  int mode;
  bool fixed;
  if (!b || !pf_mode(pub, mode, fixed)) return MOE_EINVAL;
  const moe_layer_geom& g = b->geom;
  if (g.gate_up_type != MOE_NVFP4 || g.down_type != MOE_NVFP4) return MOE_EUNSUPPORTED;
  if (g.H % 256 != 0 || g.I % 256 != 0) return MOE_EUNSUPPORTED;
  return MOE_OK;
}

}  // namespace

size_t moe_prefill_workspace_bytes(const moe_bank* b, int32_t T, int32_t mode) {
  if (pf_check(b, mode) != MOE_OK || T < 1) return 0;
  if ((int64_t)T * b->geom.top_k > (int64_t)(1 << 30)) return 0;
  int m;
  bool fixed;
  pf_mode(mode, m, fixed);
  return pf_layout(b->geom, T, m, pf_fp4(b, m), fixed).total;
}

static int prefill_impl(const moe_bank* b, const void* x, int32_t T, const int32_t* ids, const float* w, int32_t pub,
                        void* out, void* ws, size_t ws_bytes, void* stream, bool export_i16) {
  int st = pf_check(b, pub);
  if (st) return st;
  int mode;
  bool fixed;
  pf_mode(pub, mode, fixed);
  if (T < 0) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  if (!x || !ids || !w || !out || !ws) return MOE_EINVAL;
  if (!aligned(x, 16) || !aligned(out, 8) || !aligned(ids, 4) || !aligned(w, 4) || !aligned(ws, 256))
    return MOE_EINVAL;
  const moe_layer_geom& g = b->geom;
  if ((int64_t)T * g.top_k > (int64_t)(1 << 30)) return MOE_EINVAL;
  const PfLayout L = pf_layout(g, T, mode, pf_fp4(b, mode), fixed);
  if (ws_bytes < L.total) return MOE_EINVAL;
  uint8_t* base = static_cast<uint8_t*>(ws);
  PfParams p;
  std::memset(&p, 0, sizeof(p));
  p.H = g.H; p.I = g.I; p.E = g.E; p.K = g.top_k; p.T = T; p.RT = T * g.top_k;
  p.mode = mode;
  p.glu = g.glu;
  p.rb_gu = b->rb_gu; p.rb_dn = b->rb_dn;
  p.gu_bank = b->gu; p.dn_bank = b->dn; p.scales = b->scales;
  p.x = static_cast<const uint16_t*>(x);
  p.ids = ids;
  p.w = w;
  p.out = static_cast<uint16_t*>(out);
  p.err = reinterpret_cast<uint32_t*>(base + L.err);
  p.off = reinterpret_cast<int*>(base + L.off);
  p.perm = reinterpret_cast<int*>(base + L.perm);
  p.bcnt = reinterpret_cast<int*>(base + L.bcnt);
  p.xq = base + L.xq;
  p.x16 = reinterpret_cast<uint16_t*>(base + L.x16);
  p.x16lo = reinterpret_cast<uint16_t*>(base + L.x16lo);
  p.i16 = reinterpret_cast<uint16_t*>(base + L.i16);
  p.y = reinterpret_cast<float*>(base + L.y);
  // W4A4 runs on the block-scaled FP4 tensor cores when the bank has its TMA maps
  if (pf_fp4(b, mode)) {
    // the FP4 GEMMs number their tiles in int: (row blocks) x (column blocks) stays below 2^31
    const long long rbmax = (long long)T * g.top_k / 128 + g.E;
    const long long cbmax = g.I / 64 > g.H / 128 ? g.I / 64 : g.H / 128;
    if (rbmax * cbmax >= (1LL << 31)) return MOE_EUNSUPPORTED;
    p.inv = reinterpret_cast<int*>(base + L.inv);
    p.xs = base + L.xs;
    p.ysum = fixed ? nullptr : p.y;
    Pf4Params q;
    std::memset(&q, 0, sizeof(q));
    // weight boxes of 128 rows (a gate_up tile loads its 128 gate and 128 up rows)
    q.map_wdn = b->map_dn; q.map_wdns = b->map_dns;
    q.H = g.H; q.I = g.I; q.E = g.E; q.K = g.top_k; q.T = T; q.RT = T * g.top_k;
    q.glu = g.glu;
    q.export_i16 = export_i16 ? 1 : 0;
    q.scales = b->scales; q.ids = ids; q.w = w;
    q.err = p.err; q.off = p.off; q.perm = p.perm;
    q.xs = base + L.xs;
    q.in4 = base + L.in4;
    q.i16 = p.i16;
    q.y = p.y;
    q.out = p.out;
    q.fixed = fixed ? 1 : 0;
    const uint64_t rbx = (uint64_t)(g.H / 2 + g.H / 16), rbi = (uint64_t)(g.I / 2 + g.I / 16);
    if (!map_byte_rows(&q.map_wgu, b->gu, (uint64_t)g.E * 2 * g.I, rbx, 128, 128, true) ||
        !map_byte_rows(&q.map_wgus, b->gu, (uint64_t)g.E * 2 * g.I, rbx, 16, 128) ||
        !map_byte_rows(&q.map_xs, q.xs, (uint64_t)q.RT, rbx, 128, 128, true) ||
        !map_byte_rows(&q.map_xss, q.xs, (uint64_t)q.RT, rbx, 16, 128) ||
        !map_byte_rows(&q.map_in, q.in4, (uint64_t)q.RT, rbi, 128, 128, true) ||
        !map_byte_rows(&q.map_ins, q.in4, (uint64_t)q.RT, rbi, 16, 128)) {
      std::snprintf(g_cuda_err, sizeof(g_cuda_err), "prompt path: tensor map encode failed");
      return MOE_ECUDA;
    }
    p.x16 = nullptr;   // the fp16 operand of the kind::f16 GEMMs is not needed
    cudaError_t e = launch_prefill(p, static_cast<cudaStream_t>(stream), &q);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "prefill launch");
  }
  cudaError_t e = launch_prefill(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "prefill launch");
}

int moe_prefill_grouped(const moe_bank* b, const void* x, int32_t T, const int32_t* ids, const float* w,
                        int32_t mode, void* out, void* ws, size_t ws_bytes, void* stream) {
  return prefill_impl(b, x, T, ids, w, mode, out, ws, ws_bytes, stream, false);
}

int moe_debug_prefill_stages(const moe_bank* b, const void* x, int32_t T, const int32_t* ids, const float* w,
                             int32_t mode, void* out, void* ws, size_t ws_bytes, void* stream, void* xq,
                             int32_t* off, int32_t* perm, void* i16) {
  int st = prefill_impl(b, x, T, ids, w, mode, out, ws, ws_bytes, stream, true);
  if (st || T == 0) return st;
  const moe_layer_geom& g = b->geom;
  bool fixed;
  pf_mode(mode, mode, fixed);
  const PfLayout L = pf_layout(g, T, mode, pf_fp4(b, mode), fixed);
  const uint8_t* base = static_cast<const uint8_t*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t RT = (size_t)T * g.top_k;
  cudaError_t e = cudaSuccess;
  const size_t xq_bytes = (mode == PF_W4A4) ? (size_t)T * (g.H / 2 + g.H / 16)
                          : (mode == PF_W4A8) ? (size_t)T * (g.H / 32) * 36 : 2 * (size_t)T * g.H;
  if (xq) e = cudaMemcpyAsync(xq, base + (mode == PF_FP16 ? L.x16 : L.xq), xq_bytes, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && off) e = cudaMemcpyAsync(off, base + L.off, 4 * ((size_t)g.E + 1), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && perm) e = cudaMemcpyAsync(perm, base + L.perm, 4 * RT, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && i16) e = cudaMemcpyAsync(i16, base + L.i16, 2 * RT * g.I, cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "prefill debug export");
}

int moe_linear(int32_t type, const void* rows, int32_t N, int32_t K, const float* row_scale, const void* x,
               int32_t T, void* out, uint32_t* dev_err, void* stream) {
  if (T == 0) return MOE_OK;
  if (!rows || !x || !out || N < 1 || K < 32 || T < 0) return MOE_EINVAL;
  if (type < MOE_BF16 || type > MOE_F32) return MOE_EINVAL;
  if (is_float_w(type)) return MOE_EUNSUPPORTED;
  if (T > MOE_LINEAR_MAX_T) return MOE_EUNSUPPORTED;
  const int rb = row_bytes_of(type, K);
  if (rb == 0) return MOE_EINVAL;
  if (!aligned(rows, 16) || !aligned(x, 16) || !aligned(out, 2) || (row_scale && !aligned(row_scale, 4)) ||
      (dev_err && !aligned(dev_err, 4)))
    return MOE_EINVAL;
  LinParams p;
  std::memset(&p, 0, sizeof(p));
  p.type = type; p.N = N; p.K = K; p.T = T; p.rb = rb;
  p.rows = static_cast<const uint8_t*>(rows);
  p.row_scale = row_scale;
  p.x = static_cast<const uint16_t*>(x);
  p.out = static_cast<uint16_t*>(out);
  p.err = dev_err;
  if (!plan_linear(p)) return MOE_EUNSUPPORTED;
  cudaError_t e = launch_linear(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "linear");
}

int moe_debug_tc_gemm(const void* A, const void* B, int32_t K, int32_t N, float* D, int32_t* dev_err,
                      void* stream) {
  if (!A || !B || !D || !dev_err || K <= 0 || K % 64 != 0 || N < 16 || N > 256 || N % 16 != 0) return MOE_EINVAL;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 4) || !aligned(dev_err, 4)) return MOE_EINVAL;
  cudaError_t e = launch_tc_gemm_check(static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(B), K, N, D,
                                       dev_err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "tc_gemm");
}

int moe_debug_wait_timeout(int32_t mode, int32_t limit, uint32_t* dev_err, void* stream) {
  if (!dev_err || !aligned(dev_err, 4) || (mode != 0 && mode != 1)) return MOE_EINVAL;
  if (limit < 1 || limit > MOE_DEBUG_WAIT_MAX) return MOE_EINVAL;
  cudaError_t e = launch_wait_timeout(mode, (uint32_t)limit, dev_err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "wait_timeout");
}

int moe_debug_fp4_gemm(const void* A, const void* scale_A, const void* B, const void* scale_B, int32_t K,
                       int32_t N, float* D, int32_t* dev_err, void* stream) {
  if (!A || !scale_A || !B || !scale_B || !D || !dev_err) return MOE_EINVAL;
  if (K < 256 || K % 256 != 0 || N < 16 || N > 256 || N % 16 != 0) return MOE_EINVAL;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(scale_A, 16) || !aligned(scale_B, 16) || !aligned(D, 4) ||
      !aligned(dev_err, 4))
    return MOE_EINVAL;
  cudaError_t e = launch_fp4_gemm_check(static_cast<const uint8_t*>(A), static_cast<const uint8_t*>(scale_A),
                                        static_cast<const uint8_t*>(B), static_cast<const uint8_t*>(scale_B), K, N, D,
                                        dev_err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "fp4_gemm");
}

int moe_debug_decode_stages(const moe_bank* b, const void* x, int32_t T, const int32_t* ids, const float* w,
                            void* out, void* ws, size_t ws_bytes, void* stream, void* x_blocks, float* inter,
                            void* inter_blocks) {
  if (!b) return MOE_EINVAL;
  const Shape sh = decode_shape(b->geom);
  if (T > sh.t_chunk) return MOE_EINVAL;
  int st = decode_impl(b, x, T, ids, w, out, ws, ws_bytes, stream, nullptr);
  if (st || T == 0) return st;
  const moe_layer_geom& g = b->geom;
  const WsLayout L = ws_layout(g, T);
  uint8_t* base = static_cast<uint8_t*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  const int64_t RT = (int64_t)T * g.top_k;
  if (x_blocks && !is_float_w(g.gate_up_type))
    e = launch_export_q8(reinterpret_cast<int8_t*>(base + L.xq), reinterpret_cast<float*>(base + L.xd),
                         reinterpret_cast<uint16_t*>(base + L.xsh), (int64_t)T * (g.H / 32),
                         static_cast<uint8_t*>(x_blocks), s);
  if (e == cudaSuccess && inter)
    e = cudaMemcpyAsync(inter, base + L.inter, 4 * (size_t)RT * g.I, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && inter_blocks && !is_float_w(g.down_type))
    e = launch_export_q8(reinterpret_cast<int8_t*>(base + L.iq), reinterpret_cast<float*>(base + L.id),
                         reinterpret_cast<uint16_t*>(base + L.ish), RT * (g.I / 32),
                         static_cast<uint8_t*>(inter_blocks), s);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "debug export");
}

}  // extern "C"
