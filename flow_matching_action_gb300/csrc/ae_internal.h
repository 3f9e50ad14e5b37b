// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>
#include <vector>

#include "../../include/ae.h"

namespace ae {

typedef __nv_bfloat16 bf16;

// Device-side error codes written to the context's status word.
enum DeviceError : int {
  kDevOk = 0,
  kDevBounds = 1,   // an index failed its bounds check; the access was skipped
  kDevTimeout = 2,  // a bounded wait gave up
};

struct Dims {
  int L, D, F, Hq, Hkv, dh, A, H;
  double eps, theta, tmin, tmax;
  int dtype;
  int C;  // width of the VLM hidden states projected by ae_bind_context (0: none)
  int qdim() const { return Hq * dh; }
  int kvdim() const { return Hkv * dh; }
  int qkvdim() const { return (Hq + 2 * Hkv) * dh; }
};

// adaRMS modulation table for one n_steps: every (step, layer, norm) triple of
// (scale, shift, gate) vectors plus the final norm's (scale, shift).
struct TimeTable {
  int n_steps = 0;
  float* mod = nullptr;  // [S][L][2][3D]
  float* fin = nullptr;  // [S][2D]
  float* act = nullptr;  // [S][2][D] sinusoid / hidden of the time MLP (scratch)
  float* c = nullptr;    // [S][D] time-MLP output
  float* fold = nullptr; // bf16 path: [S][L][(Hq+2Hkv)dh + 2F] shift W^T of the QKV and gate/up GEMMs
};

struct BindState {
  int batch = -1;                       // -1: nothing bound
  const void* pk = nullptr;             // borrowed prefix K
  const void* pv = nullptr;             // borrowed prefix V
  int64_t total_rows = 0;               // rows per layer of pk / pv
  int max_phys_rows = 0;                // longest request of the binding
  CUtensorMap map_pk, map_pv;           // bf16 path: TMA views of pk / pv, boxes 64 rows x 64
  CUtensorMap map_pk3, map_pv3;         // the same as boxes of 64 rows x head_dim (all column blocks)
  std::vector<int> lens;                // physical rows of every request
};

}  // namespace ae

struct ae_ctx {
  ae::Dims d;
  int max_batch = 0, max_rows = 0;
  cudaStream_t stream = nullptr;
  int device = 0, sm_count = 0;

  // Library-owned weights (type T = bf16 or float per d.dtype).
  void* w_in = nullptr;   // [D, A]
  void* b_in = nullptr;   // [D]
  void* w_t1 = nullptr;   // [D, D]
  void* b_t1 = nullptr;
  void* w_t2 = nullptr;
  void* b_t2 = nullptr;
  void* w_modf = nullptr; // [2D, D]
  void* b_modf = nullptr; // [2D]
  void* w_out = nullptr;  // [A, D]
  void* b_out = nullptr;  // [A]
  void* w_qkv = nullptr;  // [L][(Hq+2Hkv)dh, D]  rows: q heads | k heads | v heads
  void* w_o = nullptr;    // [L][D, Hq dh]
  void* w_gu = nullptr;   // [L][2F, D]           rows: gate | up
  void* w_d = nullptr;    // [L][D, F]
  void* w_mod = nullptr;  // [L][2][3D, D]
  void* b_mod = nullptr;  // [L][2][3D]
  // fp8 weights (ae_config.weight_format AE_WEIGHTS_FP8_E4M3): w_qkv, w_o,
  // w_gu and w_d hold e4m3 codes (uint8, same packed layout) instead of bf16,
  // and w_scale_* the dequantization factor of each packed row's tensor.
  bool w_fp8 = false;
  float* w_scale_qkv = nullptr;  // [L][(Hq+2Hkv)dh]
  float* w_scale_o = nullptr;    // [L][D]
  float* w_scale_gu = nullptr;   // [L][2F]
  float* w_scale_d = nullptr;    // [L][D]
  float* fp8_tensor_scale = nullptr;  // [L][7] factor of wq, wk, wv, wo, wg, wu, wd
  // Context projection (ctx_dim > 0): per layer [K rows | V rows] of [2 Hkv dh, C];
  // rows of every head as rotation pairs when ctx_tc (the tensor-core path).
  void* w_ctx = nullptr;
  bool ctx_tc = false;        // context projection on the tensor cores
  void* ctx_k = nullptr;      // [L][rows][Hkv dh] T: projected K of the bound context
  void* ctx_v = nullptr;      // [L][rows][Hkv dh] T
  float2* ctx_rope = nullptr; // [max_batch * max_rows][dh/2] (cos, sin) at each valid row's position
  float* ctx_tmp = nullptr;   // [max_batch * max_rows][2 Hkv dh] fp32 (SIMT projection)
  CUtensorMap map_wctx;       // w_ctx, boxes 128 rows x 64

  // Scratch, sized for max_batch * H rows.
  float* h = nullptr;        // [M, D]    residual stream
  void* y = nullptr;         // [M, D]    T, normalized + modulated activations
  float* qkv_f = nullptr;    // [M, qkv]  fp32 projection output
  void* qkv = nullptr;       // [M, qkv]  T, after RoPE
  void* o = nullptr;         // [M, Hq dh] T, attention output
  float* gu_f = nullptr;     // [M, 2F]   fp32 gate/up output
  void* m = nullptr;         // [M, F]    T, GeGLU output

  // Bind tables.
  int* valid_idx = nullptr;  // [max_batch][max_rows] physical row of each valid row
  int* n_valid = nullptr;    // [max_batch]
  float2* rope_cs = nullptr; // [max_batch][H][dh/2] (cos, sin) at the action positions
  ae::BindState bind;

  std::vector<ae::TimeTable> tables;

  // Sticky device status: host-mapped so it can be read without a sync.
  int* status_host = nullptr;
  int* status_dev = nullptr;

  float* dump = nullptr;
  size_t dump_cap = 0;

  // bf16 tensor-core path: TMA descriptors of the stacked per-layer weights
  // (rows of layer l start at l * rows-per-layer) and its extra scratch.
  bool fast = false;
  bool pdl = false;        // chain kernels by programmatic dependent launch
  bool use_graph = false;  // capture and replay the launch sequence
  CUtensorMap map_qkv, map_o, map_gu, map_d;   // weights, boxes 128 rows x 64
  CUtensorMap map_y, map_oact, map_mact;        // bf16 activations, boxes act_box_rows x 64
  CUtensorMap map_yq;                           // the QKV GEMM's operand, boxes act_box_rows_q x 64
  CUtensorMap map_attn_o;                       // attention O partials (fp32)
  CUtensorMap map_attn_o16;                     // the same buffer as bf16 partials of O / l
  CUtensorMap map_qkv_act;                      // q|k|v activations, boxes 16 rows x 64
  CUtensorMap map_qtile;                        // the same, boxes q_box_rows rows x 64 (attention query tiles)
  int q_box_rows = 16;
  int act_box_rows = 0, act_box_rows_q = 0;
  float* sumsq = nullptr;    // [D/128][M] sums of h^2 per 128-feature tile (adaRMS folded into GEMMs)
  float* attn_o = nullptr;   // attention partials
  float2* attn_ml = nullptr;
  float* x = nullptr;        // [M, A] flow state while a captured graph runs

  // The whole launch sequence of one ae_sample, captured once per binding and
  // n_steps and replayed (kernels chained by programmatic dependent launch).
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t graph_exec = nullptr;
  int64_t graph_launches = 0;
  struct GraphKey {
    int batch = -1, n_steps = 0, max_phys_rows = 0;
    const void *pk = nullptr, *pv = nullptr;
    int64_t total_rows = 0;
    const float* dump = nullptr;
    std::vector<int> lens;  // the attention work split depends on every request's length
    bool operator==(const GraphKey& o) const {
      return batch == o.batch && n_steps == o.n_steps && max_phys_rows == o.max_phys_rows &&
             pk == o.pk && pv == o.pv && total_rows == o.total_rows && dump == o.dump && lens == o.lens;
    }
  } graph_key;

  int64_t launches_sample = 0, launches_bind = 0, device_bytes = 0;
  std::vector<void*> allocations;
  std::string last_msg;
};

namespace ae {

// Launch a kernel; with pdl, as a programmatic dependent of the previous
// kernel of the stream (it may start early and waits in griddepcontrol.wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Parameters of the bind kernel; every request's physical row range travels
// by value with the launch (ranges may coincide: samples sharing one prefix).
struct BindArgs {
  int batch;
  int max_rows;
  int lo[AE_MAX_BATCH], hi[AE_MAX_BATCH];  // request b owns physical rows [lo[b], hi[b])
  const uint8_t* mask;
  int* valid_idx;
  int* n_valid;
  float2* rope_cs;
  int H, half_dh;
  double theta;
  int* status;
};

// Launch wrappers (ae_simt.cu).  Each returns the number of kernels it enqueued.
int launch_bind(const BindArgs& a, cudaStream_t s);
int launch_time_table(const ae_ctx* c, TimeTable& t, cudaStream_t s);
int launch_step_simt(ae_ctx* c, const TimeTable& t, int step, float* x, cudaStream_t s);
int launch_attn_bf16(ae_ctx* c, int layer, cudaStream_t s);
cudaError_t launch_final_bf16(ae_ctx* c, const TimeTable& t, int step, float* x, cudaStream_t s,
                              bool pdl);

// ---- tensor-core GEMM (ae_gemm_tc.cu)
enum EMode : int { kEPartial = 0, kEQkvRope = 1, kEGeglu = 2, kEResid = 3 };
struct TcGemmArgs {
  int M, N, K;          // tokens, output features, reduction length
  int w_row0;           // first row of this layer's matrix in the stacked weight
  int w_next_row0;      // first row of the matrix to prefetch into L2 (-1: none)
  int tok_tile, n_tiles, tok_tiles, ksplit, kb_total, stages, tmem_cols;
  int tok_half;         // first token column of the second epilogue half (multiple of 16)
  int xbulk;            // split K: partials sent by bulk copies (1) or per-thread remote stores (0)
  int act_rows;         // rows of the operand map's token box (0: tok_tile); a single short tile loads only its valid rows
  int act_row0;         // row of the operand map where token 0 sits (a layer of a stacked operand)
  // z_count > 1 runs that many GEMMs of this shape in one launch (gridDim.y):
  // the z-th reads weight rows + z * z_w_rows, operand rows + z * z_act_rows
  // and writes out_bf16 + z * z_out (kEQkvRope only)
  int z_count, z_w_rows, z_act_rows;
  long z_out;
  int e_mode;           // kEQkvRope, kEGeglu or kEResid
  // kEQkvRope / kEGeglu: the operand is bf16(h * (1 + scale)); adaRMS is folded in
  const float* ss_in;   // [n_ss][M] sums of h^2 per 128 features of the operand's rows
  int n_ss, norm_dim;   // D / 128, D; n_ss == 0: no norm (a plain projection)
  float eps;
  const float* fold;    // [N] shift W^T of this layer and flow step (nullptr: none)
  // fp8 weights: dequantization factor of every row of the stacked weight
  // (row w_row0 + z * z_w_rows + n); unused by the bf16-weight kernels
  const float* w_scale;
  bf16* out_bf16;       // kEQkvRope: [M][N]; kEGeglu: [M][N/2]
  const float2* rope_cs;
  int dh, n_rot_heads;
  // kEResid: h += gate * acc, then the next GEMM's operand and its sums of squares
  float* h;                 // [M][N] residual stream, updated in place
  const float* gate;        // [N]
  const float* scale_next;  // [N], or nullptr when no GEMM follows
  bf16* a_out;              // [M][N] bf16(h * (1 + scale_next))
  float* ss_out;            // [N/128][M]
  int* status;
};
struct GemmPlan {
  int N, K, n_tiles, tok_tiles, tok_tile, kb_total, ksplit, tmem_cols, stages, grid;
  int xbulk;  // split K: the fp32 tile fits the drained pipeline buffers, partials go by bulk copy
  int wf;     // 1: the weights are e4m3 codes (the kernels that widen them to bf16)
  size_t smem;
};
size_t tc_gemm_smem_bytes(int stages, int tok_tile);
// Split-K plan of k_tc_gemm: the splits of a tile form one cluster (<= 16 CTAs),
// no more splits than keep every cluster of the launch resident at once.
// retile: an unsplit plan that leaves SMs idle may use more, shorter token
// tiles (the operand's TMA box must then follow the plan's tok_tile).
// exact_split > 0: exactly that many K splits whatever M is (the sum order over
// K, and so the rounding of every output, then does not depend on M).
// wf = 1: e4m3 weights (an 8 KB staging buffer more per pipeline stage).
GemmPlan plan_gemm_cl(int N, int K, int M, int sm_count, int max_split = 0, bool retile = false,
                      int exact_split = 0, int wf = 0);
cudaError_t gemm_kernel_setup();
// The e4m3-weight instantiations of k_tc_gemm (ae_gemm_fp8.cu).
typedef void (*GemmKernel)(const CUtensorMap, const CUtensorMap, const TcGemmArgs);
GemmKernel gemm_kernel_fp8(int ew, int mode, int xp);
cudaError_t gemm_kernel_setup_fp8();
// Per-tensor e4m3 quantization of a packed, layer-stacked bf16 weight
// [L][rows][K] into codes [L][rows][K] (ae_gemm_fp8.cu).  The rows of one
// layer belong to its tensors as `groups` says: tensors t0, t0 + 1, t0 + 2 over
// the row ranges [0, b1), [b1, b2), [b2, rows) (kind 0; b1 = b2 = rows for a
// single tensor), or alternately by row parity (kind 1: even rows t0, odd
// rows t0 + 1).  Tensor t of layer l is slot l * 7 + t of amax / scale.
struct RowGroups {
  int rows, kind, b1, b2, t0;
};
// amax[l * 7 + t] = max |w| over the tensor (amax zeroed by the caller)
cudaError_t launch_tensor_amax(const bf16* W, int L, int K, RowGroups g, float* amax, cudaStream_t s);
// s = 448 / amax (1 when amax == 0) and r = 1 / s for n slots, fp32 round-to-nearest
cudaError_t launch_tensor_scales(const float* amax, int n, float* s_out, float* r_out, cudaStream_t st);
// codes = e4m3(w * s) (round to nearest even, saturating) and row_r[row] = r of the row's tensor
cudaError_t launch_quantize_e4m3(const bf16* W, int L, int K, RowGroups g, const float* s_slot,
                                 const float* r_slot, uint8_t* codes, float* row_r, cudaStream_t st);
// launch_fold_shift over e4m3 codes: fold = r_row[n] * sum_k e4m3(W8[n][k]) shift[k]
cudaError_t launch_fold_shift_e4m3(const uint8_t* W8, const float* row_r, int N, int D, const float* mod, int S,
                                   int L, int j, float* fold, int nf, int off, cudaStream_t s);
cudaError_t launch_tc_gemm(const CUtensorMap& wmap, const CUtensorMap& amap, const GemmPlan& p,
                           TcGemmArgs a, cudaStream_t s, bool pdl);
// h = emb (prefill input); aout = bf16(h * (1 + scale)); ss_out [D/128][M] sums of h^2.
cudaError_t launch_embed_norm(const bf16* emb, int M, int D, float* h, const float* scale, bf16* aout,
                              float* ss_out, cudaStream_t s, bool pdl);
// h = x W_in^T + b_in; aout = bf16(h * (1 + scale)); ss_out [D/128][M] sums of h^2.
cudaError_t launch_inproj_norm(const float* x, const bf16* w_in, const bf16* b_in, int M, int D, int A,
                               float* h, const float* scale, bf16* aout, float* ss_out, cudaStream_t s,
                               bool pdl);
// fold[s][l][off + n] = sum_k W[l][n][k] * mod[s][l][j][shift][k] for every step and layer.
cudaError_t launch_fold_shift(const bf16* W, int N, int D, const float* mod, int S, int L, int j, float* fold,
                              int nf, int off, cudaStream_t s);
// ---- tensor-core attention (ae_attn_tc.cu)
struct AttnArgs {
  const bf16* qkv;        // [M][(Hq + 2 Hkv) dh] after RoPE
  const bf16* pk;         // this layer's prefix K [total_rows][Hkv dh]
  const bf16* pv;
  long total_rows;
  const int* valid_idx;   // [batch][max_rows]
  const int* n_valid;     // [batch]
  int max_rows;           // row stride of valid_idx
  int plan_rows;          // longest physical prefix of the bound requests (work split bound)
  const int* host_lens;   // host copy of every request's physical row count, for the work split; may be null
  int layer_row0;         // first row of this layer in the prefix K/V maps
  int batch, H, Hq, Hkv, dh;
  float scale;
  int q_tiles, chunks_per_cta, max_splits;  // set by the planner
  int max_units;          // cap on work units (0: none), for fixed-size scratch
  int q_box;              // rows of a query-tile TMA box (64, 32 or 16; divides the padded head length)
  float* part_o;          // [units][128][dh] fp32 O, or (o16) bf16 O / l
  float2* part_ml;        // [units][128]
  int o16;                // partials stored as bf16 rows of O / l (omap: bf16 boxes of 128 rows x 64)
  int* status;
};
size_t attn_part_units(int max_batch, int H, int Hq, int Hkv, int max_rows, int sm_count);
// Work units the planner would use (within a.max_units when it is set; a
// result above a.max_units means the cap cannot be met).
size_t attn_plan_units(AttnArgs a, int sm_count);
cudaError_t attn_kernel_setup();
// qmap: bf16 [maxM, (Hq + 2 Hkv) dh] view of the q|k|v activations, boxes a.q_box rows x 64.
// kmap, vmap: bf16 [L * total_rows, Hkv dh] views of the bound prefix K / V, boxes 64 rows x 64.
// omap: fp32 [units * 128, dh] view of part_o, boxes of 128 rows x 32 columns, 128-byte swizzle.
// omap16: bf16 view of the same partials (make_attn_o16_map), or nullptr (fp32
// partials through omap).
cudaError_t launch_attn_tc(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& kmap3, const CUtensorMap& vmap3,
                           const CUtensorMap& omap, const CUtensorMap* omap16, AttnArgs a, bf16* o, int sm_count,
                           cudaStream_t s, bool pdl);
cudaError_t make_bf16_map(CUtensorMap* map, const void* ptr, long rows, long cols, int box_rows);
// fp32 [d2][d1][d0] view with boxes {32, box1, 1}, 128-byte swizzle (split-K partials)
cudaError_t make_kv3d_map(CUtensorMap* map, const void* ptr, long rows, long kvdim, int dh);
cudaError_t make_f32_3d_map(CUtensorMap* map, const void* ptr, long d0, long d1, long d2, int box1);
cudaError_t make_attn_o_map(CUtensorMap* map, float* part_o, size_t units, int dh);
// bf16 [units * 128, dh] view of part_o, boxes of 128 rows x 64 columns, 128-byte swizzle
cudaError_t make_attn_o16_map(CUtensorMap* map, float* part_o, size_t units, int dh);

// ---- context projection (ae_bind_context)
// ctx_rope[valid row of request b at position i] = (cos, sin)(i theta^(-2j/dh)).
int launch_ctx_rope(const int* valid_idx, const int* n_valid, int batch, int max_rows, int half_dh, double theta,
                    float2* ctx_rope, cudaStream_t s);
// SIMT projection of one layer: [K | V] = hidden W_ctx^T for all rows, then the
// valid rows rotated (K) and stored as T into k_out / v_out [rows][Hkv dh].
int launch_ctx_project_simt(const ae_ctx* c, const void* hidden_l, int64_t rows, const void* w_l, void* k_out,
                            void* v_out, cudaStream_t s);
// Tensor-core projection of every layer (bf16, Hkv dh % 128 == 0): two GEMMs a layer.
int launch_ctx_project_tc(ae_ctx* c, const void* hidden, int64_t rows, cudaStream_t s, cudaError_t* err);

// ---- bf16 path driver (ae_fast.cu)
bool fast_path_supported(const Dims& d, std::string* why);
cudaError_t fast_setup(ae_ctx* c);  // tensor maps and scratch, after the weights are packed
// one box = one token tile: box_rows for the gate/up, O and down GEMMs, box_rows_q for QKV
cudaError_t fast_activation_maps(ae_ctx* c, int box_rows, int box_rows_q);
// Attention split-KV partials supplied by the caller instead of the context's.
struct AttnScratch {
  float* part_o;
  float2* part_ml;
  int max_units;
  CUtensorMap omap;  // make_attn_o_map of part_o
};
// A prefill run of the layers (ae_prefill): embeddings replace the action
// input projection, every layer's K and V are copied out after its QKV GEMM,
// and nothing after the last layer's QKV GEMM runs.
struct PrefillOut {
  const bf16* emb;  // [M][D]
  bf16* k;          // [L][M][Hkv dh]
  bf16* v;
};
int launch_step_fast(ae_ctx* c, const TimeTable& t, int step, float* x, cudaStream_t s,
                     cudaError_t* err, const AttnScratch* attn_scratch = nullptr,
                     const PrefillOut* prefill = nullptr);
// The cached time table of n_steps, or nullptr (never allocates).
const TimeTable* find_time_table(const ae_ctx* c, int n_steps);
void attn_plan(AttnArgs& a, int sm_count);

}  // namespace ae
