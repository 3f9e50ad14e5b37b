// Driver of the bf16 tensor-core path: TMA descriptors, scratch sizing and
// the launch sequence of one flow step.
//
// One flow step (MolmoBot PR, Part 2: only the action queries and t change
// between steps; the prefix binding is reused), six kernels per layer:
//   in-proj (+ sums of squares) ->
//   per layer: [adaRMS1 folded -> merged QKV GEMM -> RoPE] -> attention ->
//              chunk combine -> [O GEMM -> gated residual] ->
//              [adaRMS2 folded -> merged gate/up GEMM -> GeGLU] ->
//              [down GEMM -> gated residual] ->
//   final adaRMS + out-proj + Euler update.
// A GEMM whose output tiles cannot fill the GPU splits K over the CTAs of a
// cluster, which sum their partials in rank order (deterministic) through
// distributed shared memory inside the same kernel.
#include <math.h>
#include <string.h>

#include <string>

#include "ae_internal.h"

namespace ae {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

// bf16 matrix [rows, K] row-major; boxes of box_rows rows x 64 columns, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* map, const void* ptr, long rows, long K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// e4m3 codes [rows, K] (one byte each); boxes of 128 rows x 128 codes, 128-byte
// swizzle (the GEMM's widening step un-swizzles them as it writes the bf16 tiles).
cudaError_t make_map_e4m3(CUtensorMap* map, const void* ptr, long rows, long K) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A stacked weight's map: bf16 boxes, or e4m3 boxes when the context quantized its block Linears.
cudaError_t make_weight_map(const ae_ctx* c, CUtensorMap* map, const void* ptr, long rows, long K) {
  return c->w_fp8 ? make_map_e4m3(map, ptr, rows, K) : make_map(map, ptr, rows, K, 128);
}

}  // namespace

bool fast_path_supported(const Dims& d, std::string* why) {
  auto no = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (d.D % 128) return no("bf16 path needs width % 128 == 0");
  if (d.F % 64) return no("bf16 path needs mlp % 64 == 0");
  if (d.qkvdim() % 128) return no("bf16 path needs (n_q_heads + 2 n_kv_heads) * head_dim % 128 == 0");
  if (d.qdim() % 64) return no("bf16 path needs n_q_heads * head_dim % 64 == 0");
  if (d.dh != 64 && d.dh != 128 && d.dh != 256) return no("bf16 path needs head_dim 64, 128 or 256");
  return true;
}

cudaError_t fast_setup(ae_ctx* c) {
  const Dims& d = c->d;
  cudaError_t e;
  const long maxM = (long)c->max_batch * d.H;
  if ((e = make_weight_map(c, &c->map_qkv, c->w_qkv, (long)d.L * d.qkvdim(), d.D)) != cudaSuccess) return e;
  if ((e = make_weight_map(c, &c->map_o, c->w_o, (long)d.L * d.D, d.qdim())) != cudaSuccess) return e;
  if ((e = make_weight_map(c, &c->map_gu, c->w_gu, (long)d.L * 2 * d.F, d.D)) != cudaSuccess) return e;
  if ((e = make_weight_map(c, &c->map_d, c->w_d, (long)d.L * d.D, d.F)) != cudaSuccess) return e;
  if ((e = make_map(&c->map_qkv_act, c->qkv, maxM, d.qkvdim(), 16)) != cudaSuccess) return e;
  // query tiles load in boxes of whole padded heads where possible (fewer TMA issues)
  const int hp = (d.H + 15) & ~15;
  c->q_box_rows = hp % 64 == 0 ? 64 : (hp % 32 == 0 ? 32 : 16);
  if ((e = make_map(&c->map_qtile, c->qkv, maxM, d.qkvdim(), c->q_box_rows)) != cudaSuccess) return e;
  if (c->ctx_tc && (e = make_map(&c->map_wctx, c->w_ctx, (long)d.L * 2 * d.kvdim(), d.C, 128)) != cudaSuccess)
    return e;
  const size_t units = attn_part_units(c->max_batch, d.H, d.Hq, d.Hkv, c->max_rows, c->sm_count);
  if ((e = make_attn_o_map(&c->map_attn_o, c->attn_o, units, d.dh)) != cudaSuccess) return e;
  return make_attn_o16_map(&c->map_attn_o16, c->attn_o, units, d.dh);
}

// bf16 [rows, kvdim] viewed as (64 columns, rows, kvdim / 64 column blocks): one box
// of 64 rows x dh columns lands as dh / 64 blocks of [64 rows][128 B], 128-byte swizzled.
cudaError_t make_kv3d_map(CUtensorMap* map, const void* ptr, long rows, long kvdim, int dh) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(kvdim / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)kvdim * 2, 128};
  cuuint32_t box[3] = {64, 64, (cuuint32_t)(dh / 64)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_bf16_map(CUtensorMap* map, const void* ptr, long rows, long cols, int box_rows) {
  return make_map(map, ptr, rows, cols, box_rows);
}

cudaError_t make_f32_3d_map(CUtensorMap* map, const void* ptr, long d0, long d1, long d2, int box1) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)d0 * 4, (cuuint64_t)d0 * d1 * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_attn_o_map(CUtensorMap* map, float* part_o, size_t units, int dh) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)dh, (cuuint64_t)(units * 128)};
  cuuint64_t strides[1] = {(cuuint64_t)dh * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, part_o, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_attn_o16_map(CUtensorMap* map, float* part_o, size_t units, int dh) {
  return make_map(map, part_o, (long)(units * 128), dh, 128);
}

cudaError_t fast_activation_maps(ae_ctx* c, int box_rows, int box_rows_q) {
  if (c->act_box_rows == box_rows && c->act_box_rows_q == box_rows_q) return cudaSuccess;
  const Dims& d = c->d;
  const long maxM = (long)c->max_batch * d.H;
  cudaError_t e;
  if ((e = make_map(&c->map_y, c->y, maxM, d.D, box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&c->map_oact, c->o, maxM, d.qdim(), box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&c->map_mact, c->m, maxM, d.F, box_rows)) != cudaSuccess) return e;
  if ((e = make_map(&c->map_yq, c->y, maxM, d.D, box_rows_q)) != cudaSuccess) return e;
  c->act_box_rows = box_rows;
  c->act_box_rows_q = box_rows_q;
  return cudaSuccess;
}

int launch_step_fast(ae_ctx* c, const TimeTable& t, int step, float* x, cudaStream_t s,
                     cudaError_t* err, const AttnScratch* attn_scratch, const PrefillOut* prefill) {
  const bool pdl = c->pdl;
  const Dims& d = c->d;
  const int B = c->bind.batch, M = B * d.H, D = d.D, F = d.F, L = d.L;
  const int nqkv = d.qkvdim(), qd = d.qdim();
  const float eps = (float)d.eps;
  const int sm = c->sm_count;
  const int wf = c->w_fp8 ? 1 : 0;
  const GemmPlan pq = plan_gemm_cl(nqkv, D, M, sm, 0, true, 0, wf);
  const GemmPlan po = plan_gemm_cl(D, qd, M, sm, 0, false, 0, wf);
  const GemmPlan pg = plan_gemm_cl(2 * F, D, M, sm, 0, false, 0, wf);
  const GemmPlan pd = plan_gemm_cl(D, F, M, sm, 0, false, 0, wf);
  // the O, gate/up and down GEMMs share one token tiling (it depends on M
  // only); the QKV GEMM may use more, shorter tiles through its own operand map
  // A single token tile loads only the M valid rows (the MMA still reads the
  // whole tile; the rows past M hold stale data and feed columns never emitted).
  const int box_m = pg.tok_tiles == 1 ? (M < pg.tok_tile ? M : pg.tok_tile) : pg.tok_tile;
  const int box_q = pq.tok_tiles == 1 ? (M < pq.tok_tile ? M : pq.tok_tile) : pq.tok_tile;
  *err = fast_activation_maps(c, box_m, box_q);
  if (*err != cudaSuccess) return 0;
  bf16* qkv = (bf16*)c->qkv;
  bf16* o = (bf16*)c->o;
  bf16* m = (bf16*)c->m;
  bf16* y = (bf16*)c->y;
  const int nf = nqkv + 2 * F;
  int n = 0;
  auto ck = [&](cudaError_t e) {
    if (e != cudaSuccess && *err == cudaSuccess) *err = e;
  };
  auto dump = [&](int l) {
    if (c->dump == nullptr) return;
    float* dst = c->dump + (((size_t)step * (L + 1) + l) * M) * D;
    ck(cudaMemcpyAsync(dst, c->h, (size_t)M * D * sizeof(float), cudaMemcpyDeviceToDevice, s));
  };
  auto mod = [&](int l, int j) { return t.mod + (((size_t)step * L + l) * 2 + j) * 3 * D; };
  auto fold = [&](int l) { return t.fold + ((size_t)step * L + l) * nf; };
  // fields shared by every GEMM of the step
  auto base_args = [&](int w_row0, int w_next_row0) {
    TcGemmArgs a = {};
    a.M = M;
    a.status = c->status_dev;
    a.w_row0 = w_row0;
    a.w_next_row0 = w_next_row0;
    a.ss_in = c->sumsq;
    a.n_ss = D / 128;
    a.norm_dim = D;
    a.eps = eps;
    a.rope_cs = c->rope_cs;
    a.dh = d.dh;
    a.n_rot_heads = d.Hq + d.Hkv;
    a.act_rows = box_m;
    return a;
  };

  // h = x W_in^T + b_in; operand of layer 0's QKV GEMM
  // The first kernel of a sample is a full dependency of whatever precedes it
  // on the stream (the bind kernel among them); every later kernel is chained
  // to its predecessor, so all of them start after the bind has completed and
  // may read its tables before griddepcontrol.wait.
  if (prefill != nullptr)
    ck(launch_embed_norm(prefill->emb, M, D, c->h, mod(0, 0), y, c->sumsq, s, false));
  else
    ck(launch_inproj_norm(x, (const bf16*)c->w_in, (const bf16*)c->b_in, M, D, d.A, c->h, mod(0, 0), y,
                          c->sumsq, s, pdl && step > 0));
  ++n;
  for (int l = 0; l < L; ++l) {
    if (prefill == nullptr) dump(l);
    const float* mod1 = mod(l, 0);
    const float* mod2 = mod(l, 1);
    const int ln = (l + 1) % L;  // whose weights each GEMM pulls into L2 ahead of use

    // adaRMS1 (folded) -> merged QKV -> RoPE
    TcGemmArgs a = base_args(l * nqkv, ln * nqkv);
    a.e_mode = kEQkvRope;
    a.act_rows = box_q;
    a.fold = fold(l);
    a.w_scale = c->w_scale_qkv;
    a.out_bf16 = qkv;
    ck(launch_tc_gemm(c->map_qkv, c->map_yq, pq, a, s, pdl));
    ++n;
    if (prefill != nullptr) {
      // this layer's K (rotated) and V: columns [Hq dh, (Hq + Hkv) dh) and the
      // next Hkv dh of the q|k|v rows, into the prefix layout [L][M][Hkv dh]
      const size_t kvd = d.kvdim(), row = (size_t)nqkv * sizeof(bf16);
      ck(cudaMemcpy2DAsync(prefill->k + (size_t)l * M * kvd, kvd * sizeof(bf16), qkv + (size_t)d.Hq * d.dh, row,
                           kvd * sizeof(bf16), M, cudaMemcpyDeviceToDevice, s));
      ck(cudaMemcpy2DAsync(prefill->v + (size_t)l * M * kvd, kvd * sizeof(bf16),
                           qkv + (size_t)(d.Hq + d.Hkv) * d.dh, row, kvd * sizeof(bf16), M,
                           cudaMemcpyDeviceToDevice, s));
      if (l + 1 == L) break;  // nothing after the last layer's K/V is an output
    }

    // attention over [valid prefix || actions]
    {
      AttnArgs at = {};
      const long lay = (long)l * c->bind.total_rows * d.kvdim();
      at.qkv = qkv;
      at.pk = (const bf16*)c->bind.pk + lay;
      at.pv = (const bf16*)c->bind.pv + lay;
      at.layer_row0 = (int)(l * c->bind.total_rows);
      at.total_rows = c->bind.total_rows;
      at.valid_idx = c->valid_idx;
      at.n_valid = c->n_valid;
      at.max_rows = c->max_rows;
      at.plan_rows = c->bind.max_phys_rows;
      at.host_lens = c->bind.lens.data();
      at.batch = B;
      at.H = d.H;
      at.Hq = d.Hq;
      at.Hkv = d.Hkv;
      at.dh = d.dh;
      at.scale = (float)(1.0 / sqrt((double)d.dh));
      at.part_o = attn_scratch ? attn_scratch->part_o : c->attn_o;
      at.part_ml = attn_scratch ? attn_scratch->part_ml : c->attn_ml;
      // the grid's work units index the partial buffers: keep them within
      // what those buffers hold (library scratch or the caller's)
      at.max_units = attn_scratch ? attn_scratch->max_units
                                  : (int)attn_part_units(c->max_batch, d.H, d.Hq, d.Hkv, c->max_rows, sm);
      at.status = c->status_dev;
      at.q_box = c->q_box_rows;
      // bf16 partials on the default path; callers' own scratch keeps fp32
      const bool o16_ok = attn_scratch == nullptr;
      ck(launch_attn_tc(c->map_qtile, c->bind.map_pk, c->bind.map_pv, c->bind.map_pk3, c->bind.map_pv3,
                        attn_scratch ? attn_scratch->omap : c->map_attn_o, o16_ok ? &c->map_attn_o16 : nullptr, at, o,
                        sm, s, pdl));
      n += 2;
    }

    // O projection -> gated residual -> operand of the gate/up GEMM (adaRMS2)
    a = base_args(l * D, ln * D);
    a.e_mode = kEResid;
    a.w_scale = c->w_scale_o;
    a.h = c->h;
    a.gate = mod1 + 2 * D;
    a.scale_next = mod2;
    a.a_out = y;
    a.ss_out = c->sumsq;
    ck(launch_tc_gemm(c->map_o, c->map_oact, po, a, s, pdl));
    ++n;

    // adaRMS2 (folded) -> merged gate/up -> GeGLU
    a = base_args(l * 2 * F, ln * 2 * F);
    a.e_mode = kEGeglu;
    a.fold = fold(l) + nqkv;
    a.w_scale = c->w_scale_gu;
    a.out_bf16 = m;
    ck(launch_tc_gemm(c->map_gu, c->map_y, pg, a, s, pdl));
    ++n;

    // down projection -> gated residual -> operand of the next layer's QKV GEMM
    a = base_args(l * D, ln * D);
    a.e_mode = kEResid;
    a.w_scale = c->w_scale_d;
    a.h = c->h;
    a.gate = mod2 + 2 * D;
    a.scale_next = l + 1 < L ? mod(l + 1, 0) : nullptr;
    a.a_out = y;
    a.ss_out = c->sumsq;
    ck(launch_tc_gemm(c->map_d, c->map_mact, pd, a, s, pdl));
    ++n;
  }
  if (prefill != nullptr) {
    ck(cudaGetLastError());
    return n;
  }
  dump(L);
  ck(launch_final_bf16(c, t, step, x, s, pdl));
  ++n;
  ck(cudaGetLastError());
  return n;
}

// Context projection on the tensor cores (ae_bind_context, MolmoBot PR,
// Part 2): per layer, K = hidden W_ck^T with RoPE at the rows' positions and
// V = hidden W_cv^T, as two GEMMs whose epilogue is the QKV epilogue without
// adaRMS (no norm, no shift): every physical row of the stacked hidden states
// [L * rows, C] is a token; masked rows yield values nothing reads.  The
// K split is fixed (kCtxSplit), not chosen from the row count: the projection
// of a valid row then sums in the same order however many masked or padded
// rows the binding has, so padded and unpadded contexts agree bitwise.
constexpr int kCtxSplit = 4;

int launch_ctx_project_tc(ae_ctx* c, const void* hidden, int64_t rows, cudaStream_t s, cudaError_t* err) {
  const Dims& d = c->d;
  const int kvd = d.kvdim(), M = (int)rows;
  const GemmPlan p = plan_gemm_cl(kvd, d.C, M, c->sm_count, 0, false, kCtxSplit);
  const int box = p.tok_tiles == 1 ? (M < p.tok_tile ? M : p.tok_tile) : p.tok_tile;
  CUtensorMap amap;
  *err = make_map(&amap, hidden, (long)d.L * M, d.C, box);
  if (*err != cudaSuccess) return 0;
  int n = 0;
  for (int part = 0; part < 2; ++part) {  // every layer's K in one launch, then every V
    TcGemmArgs a = {};
    a.M = M;
    a.status = c->status_dev;
    a.w_row0 = part * kvd;
    a.w_next_row0 = -1;
    a.n_ss = 0;  // a plain projection: no adaRMS factor
    a.norm_dim = 1;
    a.eps = 1.f;
    a.fold = nullptr;
    a.rope_cs = c->ctx_rope;
    a.dh = d.dh;
    a.n_rot_heads = part == 0 ? d.Hkv : 0;
    a.act_rows = box;
    a.act_row0 = 0;
    a.e_mode = kEQkvRope;
    a.out_bf16 = (bf16*)(part == 0 ? c->ctx_k : c->ctx_v);
    a.z_count = d.L;
    a.z_w_rows = 2 * kvd;
    a.z_act_rows = M;
    a.z_out = (long)M * kvd;
    const cudaError_t e = launch_tc_gemm(c->map_wctx, amap, p, a, s, false);
    if (e != cudaSuccess) {
      *err = e;
      return n;
    }
    ++n;
  }
  return n;
}

}  // namespace ae
