// C-ABI entry points and host runtime: argument checks, the weight packer,
// the prefix binder, the per-n_steps time-conditioning table, and the step
// loop.  No compute happens on the host; every step of the path is a kernel.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "ae_internal.h"

using ae::Dims;
using ae::TimeTable;

namespace {

thread_local std::string g_create_error;

ae_status set_msg(ae_ctx* c, ae_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c != nullptr) c->last_msg = buf;
  else g_create_error = buf;
  return st;
}

ae_status cuda_fail(ae_ctx* c, cudaError_t e, const char* what) {
  const ae_status st = (e == cudaErrorMemoryAllocation) ? AE_ERR_OOM : AE_ERR_CUDA;
  return set_msg(c, st, "%s: %s", what, cudaGetErrorString(e));
}

#define AE_CK(c, expr)                                 \
  do {                                                 \
    cudaError_t e_ = (expr);                           \
    if (e_ != cudaSuccess) return cuda_fail(c, e_, #expr); \
  } while (0)

size_t elem_size(int dtype) { return dtype == AE_DTYPE_BF16 ? 2 : 4; }

template <typename P>
ae_status alloc(ae_ctx* c, P** p, size_t bytes) {
  void* q = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaMalloc");
  c->allocations.push_back(q);
  c->device_bytes += (int64_t)bytes;
  *p = (P*)q;
  return AE_OK;
}

// Free one allocation of the context before ae_destroy (bytes: its size).
void release(ae_ctx* c, void* p, size_t bytes) {
  for (size_t i = 0; i < c->allocations.size(); ++i)
    if (c->allocations[i] == p) {
      cudaFree(p);
      c->allocations.erase(c->allocations.begin() + (long)i);
      c->device_bytes -= (int64_t)(bytes == 0 ? 16 : bytes);
      return;
    }
}

#define AE_TRY(expr)                 \
  do {                               \
    ae_status s_ = (expr);           \
    if (s_ != AE_OK) return s_;      \
  } while (0)

ae_status check_config(const ae_config* cfg) {
  if (cfg->layers <= 0 || cfg->width <= 0 || cfg->mlp <= 0 || cfg->n_q_heads <= 0 ||
      cfg->n_kv_heads <= 0 || cfg->head_dim <= 0 || cfg->action_dim <= 0 || cfg->horizon <= 0)
    return set_msg(nullptr, AE_ERR_INVALID_ARG, "every dimension must be positive");
  if (cfg->dtype != AE_DTYPE_BF16 && cfg->dtype != AE_DTYPE_F32)
    return set_msg(nullptr, AE_ERR_INVALID_ARG, "dtype must be AE_DTYPE_BF16 or AE_DTYPE_F32");
  if (cfg->n_q_heads % cfg->n_kv_heads != 0)
    return set_msg(nullptr, AE_ERR_SHAPE, "n_q_heads must be a multiple of n_kv_heads");
  if (cfg->head_dim % 32 != 0 || cfg->head_dim > 256)
    return set_msg(nullptr, AE_ERR_SHAPE, "head_dim must be a multiple of 32 and <= 256");
  if (cfg->width % 32 != 0 || cfg->mlp % 32 != 0)
    return set_msg(nullptr, AE_ERR_SHAPE, "width and mlp must be multiples of 32");
  if (!(cfg->rms_eps > 0.0) || !(cfg->rope_theta > 0.0) || !(cfg->time_min_period > 0.0) ||
      !(cfg->time_max_period > 0.0))
    return set_msg(nullptr, AE_ERR_INVALID_ARG, "eps, rope_theta and time periods must be > 0");
  if (cfg->ctx_dim < 0 || cfg->ctx_dim % 8 != 0)
    return set_msg(nullptr, AE_ERR_SHAPE, "ctx_dim must be 0 or a positive multiple of 8");
  if (cfg->weight_format != AE_WEIGHTS_AS_DTYPE && cfg->weight_format != AE_WEIGHTS_FP8_E4M3)
    return set_msg(nullptr, AE_ERR_INVALID_ARG, "weight_format must be AE_WEIGHTS_AS_DTYPE or AE_WEIGHTS_FP8_E4M3");
  if (cfg->weight_format == AE_WEIGHTS_FP8_E4M3 && cfg->dtype != AE_DTYPE_BF16)
    return set_msg(nullptr, AE_ERR_INVALID_ARG, "fp8 weights need dtype AE_DTYPE_BF16");
  return AE_OK;
}

ae_status check_weights(const ae_config* cfg, const ae_weights* w) {
  const void* globals[] = {w->w_in, w->b_in, w->w_t1, w->b_t1, w->w_t2,
                           w->b_t2, w->w_mod_f, w->b_mod_f, w->w_out, w->b_out};
  for (const void* p : globals)
    if (p == nullptr) return set_msg(nullptr, AE_ERR_INVALID_ARG, "a global weight pointer is NULL");
  const void* const* per[] = {w->wq, w->wk, w->wv, w->wo, w->wg, w->wu,
                              w->wd, w->w_mod1, w->b_mod1, w->w_mod2, w->b_mod2};
  for (const void* const* arr : per) {
    if (arr == nullptr) return set_msg(nullptr, AE_ERR_INVALID_ARG, "a per-layer weight array is NULL");
    for (int l = 0; l < cfg->layers; ++l)
      if (arr[l] == nullptr)
        return set_msg(nullptr, AE_ERR_INVALID_ARG, "per-layer weight pointer of layer %d is NULL", l);
  }
  if (cfg->ctx_dim > 0)
    for (const void* const* arr : {w->w_ck, w->w_cv}) {
      if (arr == nullptr) return set_msg(nullptr, AE_ERR_INVALID_ARG, "w_ck / w_cv is NULL while ctx_dim > 0");
      for (int l = 0; l < cfg->layers; ++l)
        if (arr[l] == nullptr)
          return set_msg(nullptr, AE_ERR_INVALID_ARG, "w_ck / w_cv pointer of layer %d is NULL", l);
    }
  return AE_OK;
}

// Copy one caller tensor into library memory (device or host source).
ae_status put(ae_ctx* c, void* dst, const void* src, size_t bytes) {
  AE_CK(c, cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, c->stream));
  return AE_OK;
}

// The weight packer: library-owned copies; Q/K/V rows and gate/up rows are
// merged into one matrix each (sglang PR #34599 item 1), every layer's two
// modulation Linears into one [2 * 3D, D] block.
ae_status pack_weights(ae_ctx* c, const ae_weights* w) {
  const Dims& d = c->d;
  const size_t es = elem_size(d.dtype);
  const size_t D = d.D, F = d.F, A = d.A, L = d.L;
  const size_t qd = d.qdim(), kvd = d.kvdim(), nqkv = d.qkvdim();
  (void)kvd;
  AE_TRY(alloc(c, &c->w_in, D * A * es));
  AE_TRY(alloc(c, &c->b_in, D * es));
  AE_TRY(alloc(c, &c->w_t1, D * D * es));
  AE_TRY(alloc(c, &c->b_t1, D * es));
  AE_TRY(alloc(c, &c->w_t2, D * D * es));
  AE_TRY(alloc(c, &c->b_t2, D * es));
  AE_TRY(alloc(c, &c->w_modf, 2 * D * D * es));
  AE_TRY(alloc(c, &c->b_modf, 2 * D * es));
  AE_TRY(alloc(c, &c->w_out, A * D * es));
  AE_TRY(alloc(c, &c->b_out, A * es));
  AE_TRY(alloc(c, &c->w_qkv, L * nqkv * D * es));
  AE_TRY(alloc(c, &c->w_o, L * D * qd * es));
  AE_TRY(alloc(c, &c->w_gu, L * 2 * F * D * es));
  AE_TRY(alloc(c, &c->w_d, L * D * F * es));
  AE_TRY(alloc(c, &c->w_mod, L * 2 * 3 * D * D * es));
  AE_TRY(alloc(c, &c->b_mod, L * 2 * 3 * D * es));
  AE_TRY(put(c, c->w_in, w->w_in, D * A * es));
  AE_TRY(put(c, c->b_in, w->b_in, D * es));
  AE_TRY(put(c, c->w_t1, w->w_t1, D * D * es));
  AE_TRY(put(c, c->b_t1, w->b_t1, D * es));
  AE_TRY(put(c, c->w_t2, w->w_t2, D * D * es));
  AE_TRY(put(c, c->b_t2, w->b_t2, D * es));
  AE_TRY(put(c, c->w_modf, w->w_mod_f, 2 * D * D * es));
  AE_TRY(put(c, c->b_modf, w->b_mod_f, 2 * D * es));
  AE_TRY(put(c, c->w_out, w->w_out, A * D * es));
  AE_TRY(put(c, c->b_out, w->b_out, A * es));
  char* qkv = (char*)c->w_qkv;
  char* gu = (char*)c->w_gu;
  char* wmod = (char*)c->w_mod;
  char* bmod = (char*)c->b_mod;
  const size_t dh = d.dh, row = D * es;
  for (size_t l = 0; l < L; ++l) {
    char* q = qkv + l * nqkv * D * es;
    if (c->fast) {
      // every head's rows as rotation pairs: packed row 2j = dim j, 2j+1 = dim j + dh/2
      const void* const* srcs[3] = {w->wq, w->wk, w->wv};
      const size_t heads[3] = {(size_t)d.Hq, (size_t)d.Hkv, (size_t)d.Hkv};
      size_t hb = 0;
      for (int part = 0; part < 3; ++part)
        for (size_t h = 0; h < heads[part]; ++h, ++hb) {
          const char* src = (const char*)srcs[part][l] + h * dh * row;
          char* dst = q + hb * dh * row;
          AE_CK(c, cudaMemcpy2DAsync(dst, 2 * row, src, row, row, dh / 2, cudaMemcpyDefault, c->stream));
          AE_CK(c, cudaMemcpy2DAsync(dst + row, 2 * row, src + dh / 2 * row, row, row, dh / 2,
                                     cudaMemcpyDefault, c->stream));
        }
    } else {
      AE_TRY(put(c, q, w->wq[l], qd * D * es));
      AE_TRY(put(c, q + qd * D * es, w->wk[l], kvd * D * es));
      AE_TRY(put(c, q + (qd + kvd) * D * es, w->wv[l], kvd * D * es));
    }
    AE_TRY(put(c, (char*)c->w_o + l * D * qd * es, w->wo[l], D * qd * es));
    char* g = gu + l * 2 * F * D * es;
    if (c->fast) {
      // gate and up rows interleaved: packed row 2j = gate j, 2j+1 = up j
      AE_CK(c, cudaMemcpy2DAsync(g, 2 * row, w->wg[l], row, row, F, cudaMemcpyDefault, c->stream));
      AE_CK(c, cudaMemcpy2DAsync(g + row, 2 * row, w->wu[l], row, row, F, cudaMemcpyDefault, c->stream));
    } else {
      AE_TRY(put(c, g, w->wg[l], F * D * es));
      AE_TRY(put(c, g + F * D * es, w->wu[l], F * D * es));
    }
    AE_TRY(put(c, (char*)c->w_d + l * D * F * es, w->wd[l], D * F * es));
    AE_TRY(put(c, wmod + (l * 2 + 0) * 3 * D * D * es, w->w_mod1[l], 3 * D * D * es));
    AE_TRY(put(c, wmod + (l * 2 + 1) * 3 * D * D * es, w->w_mod2[l], 3 * D * D * es));
    AE_TRY(put(c, bmod + (l * 2 + 0) * 3 * D * es, w->b_mod1[l], 3 * D * es));
    AE_TRY(put(c, bmod + (l * 2 + 1) * 3 * D * es, w->b_mod2[l], 3 * D * es));
  }
  if (d.C > 0) {
    // context projections, per layer [K rows | V rows] of [2 Hkv dh, C]; on the
    // tensor-core path every head's rows as rotation pairs (as for Q/K/V above)
    const size_t C = d.C, crow = C * es, kvd = d.kvdim();
    c->ctx_tc = c->fast && kvd % 128 == 0 && C % 64 == 0;
    AE_TRY(alloc(c, &c->w_ctx, L * 2 * kvd * crow));
    for (size_t l = 0; l < L; ++l) {
      char* dst0 = (char*)c->w_ctx + l * 2 * kvd * crow;
      const void* srcs[2] = {w->w_ck[l], w->w_cv[l]};
      for (int part = 0; part < 2; ++part) {
        char* dst = dst0 + part * kvd * crow;
        if (!c->ctx_tc) {
          AE_TRY(put(c, dst, srcs[part], kvd * crow));
          continue;
        }
        for (size_t h = 0; h < (size_t)d.Hkv; ++h) {
          const char* src = (const char*)srcs[part] + h * dh * crow;
          char* hd = dst + h * dh * crow;
          AE_CK(c, cudaMemcpy2DAsync(hd, 2 * crow, src, crow, crow, dh / 2, cudaMemcpyDefault, c->stream));
          AE_CK(c, cudaMemcpy2DAsync(hd + crow, 2 * crow, src + dh / 2 * crow, crow, crow, dh / 2,
                                     cudaMemcpyDefault, c->stream));
        }
      }
    }
  }
  return AE_OK;
}

// fp8 weights (MolmoBot PR, Part 3; LoongForge Pi0.5 blog, section 7): the
// packed bf16 block Linears are quantized per tensor (wq, wk, wv, wo, wg, wu,
// wd of every layer) into e4m3 codes of the same packed layout, which replace
// them; every packed row gets its tensor's dequantization factor.
ae_status quantize_weights(ae_ctx* c) {
  const Dims& d = c->d;
  const int L = d.L, D = d.D, F = d.F, qd = d.qdim(), kvd = d.kvdim(), nq = d.qkvdim();
  const int n_slots = L * 7;
  float *amax = nullptr, *sv = nullptr;
  AE_TRY(alloc(c, &amax, n_slots * sizeof(float)));
  AE_TRY(alloc(c, &sv, n_slots * sizeof(float)));
  AE_TRY(alloc(c, &c->fp8_tensor_scale, n_slots * sizeof(float)));
  AE_CK(c, cudaMemsetAsync(amax, 0, n_slots * sizeof(float), c->stream));
  struct Mat {
    void** w;
    int rows, K;
    ae::RowGroups g;
    float** row_r;
  } mats[4] = {{&c->w_qkv, nq, D, {nq, 0, qd, qd + kvd, 0}, &c->w_scale_qkv},
               {&c->w_o, D, qd, {D, 0, D, D, 3}, &c->w_scale_o},
               {&c->w_gu, 2 * F, D, {2 * F, 1, 0, 0, 4}, &c->w_scale_gu},
               {&c->w_d, D, F, {D, 0, D, D, 6}, &c->w_scale_d}};
  for (const Mat& m : mats)
    AE_CK(c, ae::launch_tensor_amax((const ae::bf16*)*m.w, L, m.K, m.g, amax, c->stream));
  AE_CK(c, ae::launch_tensor_scales(amax, n_slots, sv, c->fp8_tensor_scale, c->stream));
  for (const Mat& m : mats) {
    const size_t n = (size_t)L * m.rows * m.K;
    uint8_t* codes = nullptr;
    AE_TRY(alloc(c, &codes, n));
    AE_TRY(alloc(c, m.row_r, (size_t)L * m.rows * sizeof(float)));
    AE_CK(c, ae::launch_quantize_e4m3((const ae::bf16*)*m.w, L, m.K, m.g, sv, c->fp8_tensor_scale, codes, *m.row_r,
                                      c->stream));
    AE_CK(c, cudaStreamSynchronize(c->stream));
    release(c, *m.w, n * sizeof(ae::bf16));
    *m.w = codes;
  }
  release(c, amax, n_slots * sizeof(float));
  release(c, sv, n_slots * sizeof(float));
  c->w_fp8 = true;
  return AE_OK;
}

ae_status alloc_scratch(ae_ctx* c) {
  const Dims& d = c->d;
  const size_t es = elem_size(d.dtype);
  const size_t M = (size_t)c->max_batch * d.H;
  AE_TRY(alloc(c, &c->h, M * d.D * sizeof(float)));
  AE_TRY(alloc(c, &c->y, M * d.D * es));
  AE_TRY(alloc(c, &c->qkv_f, M * d.qkvdim() * sizeof(float)));
  AE_TRY(alloc(c, &c->qkv, M * d.qkvdim() * es));
  AE_TRY(alloc(c, &c->o, M * d.qdim() * es));
  AE_TRY(alloc(c, &c->gu_f, M * 2 * d.F * sizeof(float)));
  AE_TRY(alloc(c, &c->m, M * d.F * es));
  AE_TRY(alloc(c, &c->valid_idx, (size_t)c->max_batch * (c->max_rows > 0 ? c->max_rows : 1) * sizeof(int)));
  AE_TRY(alloc(c, &c->n_valid, (size_t)c->max_batch * sizeof(int)));
  AE_TRY(alloc(c, &c->rope_cs, (size_t)c->max_batch * d.H * (d.dh / 2) * sizeof(float2)));
  if (c->fast) {
    AE_TRY(alloc(c, &c->sumsq, (size_t)(d.D / 128) * M * sizeof(float)));
    const size_t units = ae::attn_part_units(c->max_batch, d.H, d.Hq, d.Hkv, c->max_rows, c->sm_count);
    AE_TRY(alloc(c, &c->attn_o, units * 128 * d.dh * sizeof(float)));
    AE_TRY(alloc(c, &c->attn_ml, units * 128 * sizeof(float2)));
    AE_TRY(alloc(c, &c->x, M * d.A * sizeof(float)));
  }
  if (d.C > 0) {
    // projected context K / V of up to max_batch requests of max_rows rows
    const size_t rows = (size_t)c->max_batch * (c->max_rows > 0 ? c->max_rows : 1);
    AE_TRY(alloc(c, &c->ctx_k, (size_t)d.L * rows * d.kvdim() * es));
    AE_TRY(alloc(c, &c->ctx_v, (size_t)d.L * rows * d.kvdim() * es));
    if (c->ctx_tc) AE_TRY(alloc(c, &c->ctx_rope, rows * (d.dh / 2) * sizeof(float2)));
    else AE_TRY(alloc(c, &c->ctx_tmp, rows * 2 * d.kvdim() * sizeof(float)));
  }
  return AE_OK;
}

void free_all(ae_ctx* c) {
  if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
  c->graph_exec = nullptr;
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  c->cap_stream = nullptr;
  for (void* p : c->allocations) cudaFree(p);
  c->allocations.clear();
  if (c->status_host) cudaFreeHost(c->status_host);
  c->status_host = nullptr;
}

ae_status get_table(ae_ctx* c, int n_steps, const TimeTable** out) {
  for (const TimeTable& t : c->tables)
    if (t.n_steps == n_steps) {
      *out = &t;
      return AE_OK;
    }
  const Dims& d = c->d;
  TimeTable t;
  t.n_steps = n_steps;
  const size_t S = n_steps, D = d.D, L = d.L;
  AE_TRY(alloc(c, &t.mod, S * L * 2 * 3 * D * sizeof(float)));
  AE_TRY(alloc(c, &t.fin, S * 2 * D * sizeof(float)));
  AE_TRY(alloc(c, &t.act, S * 2 * D * sizeof(float)));
  AE_TRY(alloc(c, &t.c, S * D * sizeof(float)));
  ae::launch_time_table(c, t, c->stream);
  AE_CK(c, cudaGetLastError());
  if (c->fast) {
    // adaRMS's shift folded into the QKV and gate/up GEMMs: shift W^T per step and layer
    const int nq = d.qkvdim(), ng = 2 * d.F, nf = nq + ng;
    AE_TRY(alloc(c, &t.fold, S * L * (size_t)nf * sizeof(float)));
    if (c->w_fp8) {
      AE_CK(c, ae::launch_fold_shift_e4m3((const uint8_t*)c->w_qkv, c->w_scale_qkv, nq, d.D, t.mod, n_steps, d.L, 0,
                                          t.fold, nf, 0, c->stream));
      AE_CK(c, ae::launch_fold_shift_e4m3((const uint8_t*)c->w_gu, c->w_scale_gu, ng, d.D, t.mod, n_steps, d.L, 1,
                                          t.fold, nf, nq, c->stream));
    } else {
      AE_CK(c, ae::launch_fold_shift((const ae::bf16*)c->w_qkv, nq, d.D, t.mod, n_steps, d.L, 0, t.fold, nf, 0,
                                     c->stream));
      AE_CK(c, ae::launch_fold_shift((const ae::bf16*)c->w_gu, ng, d.D, t.mod, n_steps, d.L, 1, t.fold, nf, nq,
                                     c->stream));
    }
  }
  c->tables.push_back(t);
  *out = &c->tables.back();
  return AE_OK;
}

// The launch sequence of one ae_sample on the bf16 path is captured into a CUDA
// graph the first time a (binding, n_steps, dump) combination is sampled and
// replayed afterwards; the flow state travels through c->x so the graph does
// not depend on the caller's noise / output pointers.
ae_status sample_graph(ae_ctx* c, const TimeTable& t, int n_steps, const float* noise, float* out,
                       size_t xbytes, int64_t* launches) {
  ae_ctx::GraphKey key;
  key.batch = c->bind.batch;
  key.n_steps = n_steps;
  key.max_phys_rows = c->bind.max_phys_rows;
  key.pk = c->bind.pk;
  key.pv = c->bind.pv;
  key.total_rows = c->bind.total_rows;
  key.dump = c->dump;
  key.lens = c->bind.lens;
  if (c->graph_exec == nullptr || !(key == c->graph_key)) {
    if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
    c->graph_exec = nullptr;
    AE_CK(c, cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = cudaSuccess;
    int64_t n = 0;
    for (int s = 0; s < n_steps && e == cudaSuccess; ++s)
      n += ae::launch_step_fast(c, t, s, c->x, c->cap_stream, &e);
    cudaGraph_t g = nullptr;
    const cudaError_t e2 = cudaStreamEndCapture(c->cap_stream, &g);
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess) e = cudaGraphInstantiate(&c->graph_exec, g, 0);
    if (g) cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      c->graph_exec = nullptr;
      return cuda_fail(c, e, "capturing the sample graph");
    }
    c->graph_key = key;
    c->graph_launches = n;
  }
  AE_CK(c, cudaMemcpyAsync(c->x, noise, xbytes, cudaMemcpyDeviceToDevice, c->stream));
  AE_CK(c, cudaGraphLaunch(c->graph_exec, c->stream));
  AE_CK(c, cudaMemcpyAsync(out, c->x, xbytes, cudaMemcpyDeviceToDevice, c->stream));
  *launches = c->graph_launches;
  return AE_OK;
}

ae_status sticky(const ae_ctx* c) {
  const int code = c->status_host ? *(volatile int*)c->status_host : 0;
  return code != 0 ? AE_ERR_DEVICE : AE_OK;
}

}  // namespace

namespace ae {
const TimeTable* find_time_table(const ae_ctx* c, int n_steps) {
  for (const TimeTable& t : c->tables)
    if (t.n_steps == n_steps) return &t;
  return nullptr;
}
}  // namespace ae

namespace {

// Bind `batch` requests whose physical row ranges are [lo[b], hi[b]) of prefix
// K / V with `total` rows per layer (ranges checked by the caller).
ae_status bind_ranges(ae_ctx* c, int batch, const void* prefix_k, const void* prefix_v, const int* lo,
                      const int* hi, int64_t total, const uint8_t* prefix_mask) {
  if (total > 0 && (prefix_k == nullptr || prefix_v == nullptr))
    return set_msg(c, AE_ERR_INVALID_ARG, "prefix_k / prefix_v is NULL");
  ae::BindArgs a;
  memset(&a, 0, sizeof(a));
  a.batch = batch;
  for (int b = 0; b < batch; ++b) {
    a.lo[b] = lo[b];
    a.hi[b] = hi[b];
  }
  a.max_rows = c->max_rows;
  a.mask = prefix_mask;
  a.valid_idx = c->valid_idx;
  a.n_valid = c->n_valid;
  a.rope_cs = c->rope_cs;
  a.H = c->d.H;
  a.half_dh = c->d.dh / 2;
  a.theta = c->d.theta;
  a.status = c->status_dev;
  if (c->fast && total >= 64) {
    // TMA views of the borrowed prefix K / V (host-side descriptors, no copy);
    // only chunks of 64 contiguous valid rows use them
    const long rows = (long)c->d.L * total;
    cudaError_t e = ae::make_bf16_map(&c->bind.map_pk, prefix_k, rows, c->d.kvdim(), 64);
    if (e == cudaSuccess) e = ae::make_bf16_map(&c->bind.map_pv, prefix_v, rows, c->d.kvdim(), 64);
    if (e == cudaSuccess) e = ae::make_kv3d_map(&c->bind.map_pk3, prefix_k, rows, c->d.kvdim(), c->d.dh);
    if (e == cudaSuccess) e = ae::make_kv3d_map(&c->bind.map_pv3, prefix_v, rows, c->d.kvdim(), c->d.dh);
    if (e != cudaSuccess)
      return set_msg(c, AE_ERR_INVALID_ARG,
                     "prefix_k / prefix_v cannot be described for TMA (16-byte alignment needed)");
  }
  c->launches_bind = ae::launch_bind(a, c->stream);
  AE_CK(c, cudaGetLastError());
  c->bind.batch = batch;
  c->bind.pk = prefix_k;
  c->bind.pv = prefix_v;
  c->bind.total_rows = total;
  c->bind.lens.resize(batch);
  int longest = 0;
  for (int b = 0; b < batch; ++b) {
    c->bind.lens[b] = hi[b] - lo[b];
    longest = c->bind.lens[b] > longest ? c->bind.lens[b] : longest;
  }
  c->bind.max_phys_rows = longest;
  return AE_OK;
}

}  // namespace

extern "C" {

const char* ae_status_string(ae_status s) {
  switch (s) {
    case AE_OK: return "AE_OK";
    case AE_ERR_INVALID_ARG: return "AE_ERR_INVALID_ARG";
    case AE_ERR_SHAPE: return "AE_ERR_SHAPE";
    case AE_ERR_NOT_BOUND: return "AE_ERR_NOT_BOUND";
    case AE_ERR_CUDA: return "AE_ERR_CUDA";
    case AE_ERR_DEVICE: return "AE_ERR_DEVICE";
    case AE_ERR_OOM: return "AE_ERR_OOM";
    case AE_ERR_UNSUPPORTED: return "AE_ERR_UNSUPPORTED";
  }
  return "AE_ERR_UNKNOWN";
}

ae_status ae_create(const ae_config* cfg, const ae_weights* w, int max_batch,
                    int max_prefix_rows, void* stream, ae_ctx** out) {
  if (out != nullptr) *out = nullptr;
  if (cfg == nullptr || w == nullptr || out == nullptr)
    return set_msg(nullptr, AE_ERR_INVALID_ARG, "cfg, w and out must be non-NULL");
  AE_TRY(check_config(cfg));
  AE_TRY(check_weights(cfg, w));
  if (max_batch < 1 || max_batch > AE_MAX_BATCH)
    return set_msg(nullptr, AE_ERR_SHAPE, "max_batch must be in 1..%d", AE_MAX_BATCH);
  if (max_prefix_rows < 0)
    return set_msg(nullptr, AE_ERR_SHAPE, "max_prefix_rows must be >= 0");

  int dev = 0, major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess)
    return set_msg(nullptr, AE_ERR_UNSUPPORTED, "no usable CUDA device: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return set_msg(nullptr, AE_ERR_UNSUPPORTED,
                   "built for sm_103a; the current device is compute capability %d.%d", major, minor);

  ae_ctx* c = new ae_ctx();
  c->d = Dims{cfg->layers, cfg->width, cfg->mlp, cfg->n_q_heads, cfg->n_kv_heads, cfg->head_dim,
              cfg->action_dim, cfg->horizon, cfg->rms_eps, cfg->rope_theta,
              cfg->time_min_period, cfg->time_max_period, cfg->dtype, cfg->ctx_dim};
  c->max_batch = max_batch;
  c->max_rows = max_prefix_rows;
  c->stream = (cudaStream_t)stream;
  c->device = dev;
  c->sm_count = sms;
  ae_status st = AE_OK;
  e = cudaHostAlloc((void**)&c->status_host, sizeof(int), cudaHostAllocMapped);
  if (e == cudaSuccess) {
    *c->status_host = 0;
    e = cudaHostGetDevicePointer((void**)&c->status_dev, c->status_host, 0);
  }
  if (e != cudaSuccess) st = cuda_fail(c, e, "status word");
  if (st == AE_OK && cfg->dtype == AE_DTYPE_BF16) {
    std::string why;
    if (!ae::fast_path_supported(c->d, &why)) st = set_msg(c, AE_ERR_SHAPE, "%s", why.c_str());
    // e4m3 weights stream in 128-column stages: every reduction length a multiple of 128
    if (st == AE_OK && cfg->weight_format == AE_WEIGHTS_FP8_E4M3 && (c->d.qdim() % 128 || c->d.F % 128))
      st = set_msg(c, AE_ERR_SHAPE, "fp8 weights need n_q_heads * head_dim and mlp multiples of 128");
    c->fast = true;
  }
  if (st == AE_OK) st = pack_weights(c, w);
  if (st == AE_OK && cfg->weight_format == AE_WEIGHTS_FP8_E4M3) st = quantize_weights(c);
  if (st == AE_OK) st = alloc_scratch(c);
  if (st == AE_OK && c->fast) {
    e = ae::fast_setup(c);
    if (e == cudaSuccess) e = ae::gemm_kernel_setup();
    if (e == cudaSuccess) e = ae::attn_kernel_setup();
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) st = cuda_fail(c, e, "bf16 path setup");
    // AE_GRAPH=0 / AE_PDL=0 run the same kernels launched one by one / without overlap
    const char* g = getenv("AE_GRAPH");
    const char* pd = getenv("AE_PDL");
    c->use_graph = !(g && g[0] == '0');
    c->pdl = !(pd && pd[0] == '0');
  }
  if (st == AE_OK) {
    e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) st = cuda_fail(c, e, "weight copies");
  }
  if (st != AE_OK) {
    g_create_error = c->last_msg;
    free_all(c);
    delete c;
    return st;
  }
  *out = c;
  return AE_OK;
}

void ae_destroy(ae_ctx* c) {
  if (c == nullptr) return;
  cudaStreamSynchronize(c->stream);
  free_all(c);
  delete c;
}

ae_status ae_set_stream(ae_ctx* c, void* stream) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  c->stream = (cudaStream_t)stream;
  return AE_OK;
}

ae_status ae_bind_prefix(ae_ctx* c, int batch, const void* prefix_k, const void* prefix_v,
                         const int32_t* cu_lens, const uint8_t* prefix_mask) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  if (batch < 0 || batch > c->max_batch)
    return set_msg(c, AE_ERR_SHAPE, "batch %d outside 0..%d", batch, c->max_batch);
  if (batch > 0 && cu_lens == nullptr) return set_msg(c, AE_ERR_INVALID_ARG, "cu_lens is NULL");
  int lo[AE_MAX_BATCH], hi[AE_MAX_BATCH];
  if (batch > 0) {
    if (cu_lens[0] != 0) return set_msg(c, AE_ERR_SHAPE, "cu_lens[0] must be 0");
    for (int b = 0; b < batch; ++b) {
      const int64_t len = (int64_t)cu_lens[b + 1] - cu_lens[b];
      if (len < 0) return set_msg(c, AE_ERR_SHAPE, "cu_lens decreases at request %d", b);
      if (len > c->max_rows)
        return set_msg(c, AE_ERR_SHAPE, "request %d has %lld prefix rows > max_prefix_rows %d", b,
                       (long long)len, c->max_rows);
      lo[b] = cu_lens[b];
      hi[b] = cu_lens[b + 1];
    }
  }
  return bind_ranges(c, batch, prefix_k, prefix_v, lo, hi, batch > 0 ? cu_lens[batch] : 0, prefix_mask);
}

ae_status ae_bind_prefix_shared(ae_ctx* c, int n_samples, const void* prefix_k, const void* prefix_v,
                                int32_t n_rows, const uint8_t* prefix_mask) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  if (n_samples < 0 || n_samples > c->max_batch)
    return set_msg(c, AE_ERR_SHAPE, "n_samples %d outside 0..%d", n_samples, c->max_batch);
  if (n_rows < 0 || n_rows > c->max_rows)
    return set_msg(c, AE_ERR_SHAPE, "n_rows %d outside 0..max_prefix_rows %d", n_rows, c->max_rows);
  int lo[AE_MAX_BATCH], hi[AE_MAX_BATCH];
  for (int b = 0; b < n_samples; ++b) {
    lo[b] = 0;
    hi[b] = n_rows;
  }
  return bind_ranges(c, n_samples, prefix_k, prefix_v, lo, hi, n_samples > 0 ? n_rows : 0, prefix_mask);
}

ae_status ae_bind_context(ae_ctx* c, int batch, const void* hidden, const int32_t* cu_lens,
                          const uint8_t* prefix_mask) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  const Dims& d = c->d;
  if (d.C <= 0) return set_msg(c, AE_ERR_UNSUPPORTED, "the context was created with ctx_dim 0");
  if (batch < 0 || batch > c->max_batch)
    return set_msg(c, AE_ERR_SHAPE, "batch %d outside 0..%d", batch, c->max_batch);
  if (batch > 0 && cu_lens == nullptr) return set_msg(c, AE_ERR_INVALID_ARG, "cu_lens is NULL");
  int lo[AE_MAX_BATCH], hi[AE_MAX_BATCH];
  if (batch > 0) {
    if (cu_lens[0] != 0) return set_msg(c, AE_ERR_SHAPE, "cu_lens[0] must be 0");
    for (int b = 0; b < batch; ++b) {
      const int64_t len = (int64_t)cu_lens[b + 1] - cu_lens[b];
      if (len < 0) return set_msg(c, AE_ERR_SHAPE, "cu_lens decreases at request %d", b);
      if (len > c->max_rows)
        return set_msg(c, AE_ERR_SHAPE, "request %d has %lld rows > max_prefix_rows %d", b, (long long)len,
                       c->max_rows);
      lo[b] = cu_lens[b];
      hi[b] = cu_lens[b + 1];
    }
  }
  const int64_t total = batch > 0 ? cu_lens[batch] : 0;
  if (total > 0 && hidden == nullptr) return set_msg(c, AE_ERR_INVALID_ARG, "hidden is NULL");
  // the projected K / V live in the library's buffers, laid out for this
  // binding ([L][total][Hkv dh]), and are bound like a caller's prefix
  AE_TRY(bind_ranges(c, batch, c->ctx_k, c->ctx_v, lo, hi, total, prefix_mask));
  if (total == 0) return AE_OK;
  int64_t n = 0;
  const size_t es = elem_size(d.dtype);
  if (c->ctx_tc) {
    n += ae::launch_ctx_rope(c->valid_idx, c->n_valid, batch, c->max_rows, d.dh / 2, d.theta, c->ctx_rope,
                             c->stream);
    cudaError_t e = cudaSuccess;
    n += ae::launch_ctx_project_tc(c, hidden, total, c->stream, &e);
    if (e != cudaSuccess) return cuda_fail(c, e, "context projection");
  } else {
    const size_t kv_layer = (size_t)total * d.kvdim() * es;
    for (int l = 0; l < d.L; ++l)
      n += ae::launch_ctx_project_simt(c, (const char*)hidden + (size_t)l * total * d.C * es, total,
                                       (const char*)c->w_ctx + (size_t)l * 2 * d.kvdim() * d.C * es,
                                       (char*)c->ctx_k + l * kv_layer, (char*)c->ctx_v + l * kv_layer, c->stream);
  }
  AE_CK(c, cudaGetLastError());
  c->launches_bind += n;
  return AE_OK;
}

ae_status ae_prefill(ae_ctx* c, int batch, const void* embeddings, void* out_k, void* out_v) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  if (!c->fast) return set_msg(c, AE_ERR_UNSUPPORTED, "ae_prefill runs on bf16 contexts only");
  if (batch < 1 || batch > c->max_batch)
    return set_msg(c, AE_ERR_SHAPE, "batch %d outside 1..%d", batch, c->max_batch);
  if (embeddings == nullptr || out_k == nullptr || out_v == nullptr)
    return set_msg(c, AE_ERR_INVALID_ARG, "embeddings / out_k / out_v is NULL");
  if (sticky(c) != AE_OK)
    return set_msg(c, AE_ERR_DEVICE, "a device-side check failed earlier (code %d)", *c->status_host);
  // the prefix tokens are the layer's tokens: an empty bound prefix, positions 0..H-1
  int zero[AE_MAX_BATCH] = {0};
  AE_TRY(bind_ranges(c, batch, nullptr, nullptr, zero, zero, 0, nullptr));
  const TimeTable* t = nullptr;
  AE_TRY(get_table(c, 1, &t));  // constant conditioning: the modulation biases
  ae::PrefillOut po{(const ae::bf16*)embeddings, (ae::bf16*)out_k, (ae::bf16*)out_v};
  cudaError_t e = cudaSuccess;
  c->launches_sample = ae::launch_step_fast(c, *t, 0, nullptr, c->stream, &e, nullptr, &po);
  if (e != cudaSuccess) return cuda_fail(c, e, "prefill launch");
  AE_CK(c, cudaGetLastError());
  return AE_OK;
}

ae_status ae_sample(ae_ctx* c, const float* noise, int n_steps, float* out) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  if (c->bind.batch < 0) return set_msg(c, AE_ERR_NOT_BOUND, "ae_sample before ae_bind_prefix");
  if (n_steps < 1 || n_steps > AE_MAX_STEPS)
    return set_msg(c, AE_ERR_SHAPE, "n_steps %d outside 1..%d", n_steps, AE_MAX_STEPS);
  const int B = c->bind.batch;
  if (B > 0 && (noise == nullptr || out == nullptr))
    return set_msg(c, AE_ERR_INVALID_ARG, "noise / out_actions is NULL");
  if (sticky(c) != AE_OK)
    return set_msg(c, AE_ERR_DEVICE, "a device-side check failed earlier (code %d)", *c->status_host);
  const Dims& d = c->d;
  if (c->dump != nullptr) {
    const size_t need = (size_t)n_steps * (d.L + 1) * B * d.H * d.D;
    if (need > c->dump_cap)
      return set_msg(c, AE_ERR_SHAPE, "debug dump holds %zu floats, needs %zu", c->dump_cap, need);
  }
  c->launches_sample = 0;
  if (B == 0) return AE_OK;
  const TimeTable* t = nullptr;
  AE_TRY(get_table(c, n_steps, &t));
  const size_t xbytes = (size_t)B * d.H * d.A * sizeof(float);
  int64_t n = 0;
  if (c->fast && c->use_graph) {
    AE_TRY(sample_graph(c, *t, n_steps, noise, out, xbytes, &n));
  } else {
    if (out != noise) AE_CK(c, cudaMemcpyAsync(out, noise, xbytes, cudaMemcpyDeviceToDevice, c->stream));
    for (int s = 0; s < n_steps; ++s) {
      if (c->fast) {
        cudaError_t e = cudaSuccess;
        n += ae::launch_step_fast(c, *t, s, out, c->stream, &e);
        if (e != cudaSuccess) return cuda_fail(c, e, "bf16 step launch");
      } else {
        n += ae::launch_step_simt(c, *t, s, out, c->stream);
      }
    }
  }
  c->launches_sample = n;
  AE_CK(c, cudaGetLastError());
  return AE_OK;
}

ae_status ae_set_debug_dump(ae_ctx* c, float* hidden, size_t capacity) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  c->dump = hidden;
  c->dump_cap = hidden ? capacity : 0;
  return AE_OK;
}

ae_status ae_synchronize(ae_ctx* c) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  AE_CK(c, cudaStreamSynchronize(c->stream));
  if (sticky(c) != AE_OK)
    return set_msg(c, AE_ERR_DEVICE, "device-side check failed (code %d)", *c->status_host);
  return AE_OK;
}

ae_status ae_last_error(const ae_ctx* c, char* buf, size_t n) {
  const std::string& m = c ? c->last_msg : g_create_error;
  if (buf != nullptr && n > 0) {
    const size_t k = m.size() < n - 1 ? m.size() : n - 1;
    memcpy(buf, m.data(), k);
    buf[k] = '\0';
  }
  return c ? sticky(c) : AE_OK;
}

ae_status ae_get_fp8_weight(ae_ctx* c, int layer, int which, uint8_t* codes, float* scale) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  if (!c->w_fp8) return set_msg(c, AE_ERR_UNSUPPORTED, "the context's weights are not fp8");
  const Dims& d = c->d;
  if (layer < 0 || layer >= d.L || which < 0 || which > 6)
    return set_msg(c, AE_ERR_INVALID_ARG, "layer must be in 0..%d and which in 0..6", d.L - 1);
  const size_t D = d.D, F = d.F, qd = d.qdim(), kvd = d.kvdim(), nq = d.qkvdim(), dh = d.dh;
  const uint8_t* qkv = (const uint8_t*)c->w_qkv + (size_t)layer * nq * D;
  if (codes != nullptr) {
    const cudaMemcpyKind k = cudaMemcpyDeviceToHost;
    if (which <= 2) {
      // packed head rows 2j, 2j + 1 are the head's dims j, j + dh/2
      const size_t heads = which == 0 ? d.Hq : d.Hkv;
      const size_t row0 = which == 0 ? 0 : (which == 1 ? qd : qd + kvd);
      for (size_t h = 0; h < heads; ++h) {
        const uint8_t* src = qkv + (row0 + h * dh) * D;
        uint8_t* dst = codes + h * dh * D;
        AE_CK(c, cudaMemcpy2DAsync(dst, D, src, 2 * D, D, dh / 2, k, c->stream));
        AE_CK(c, cudaMemcpy2DAsync(dst + dh / 2 * D, D, src + D, 2 * D, D, dh / 2, k, c->stream));
      }
    } else if (which == 3) {
      AE_CK(c, cudaMemcpyAsync(codes, (const uint8_t*)c->w_o + (size_t)layer * D * qd, D * qd, k, c->stream));
    } else if (which <= 5) {
      // packed rows 2j, 2j + 1 are gate row j and up row j
      const uint8_t* src = (const uint8_t*)c->w_gu + (size_t)layer * 2 * F * D + (which == 5 ? D : 0);
      AE_CK(c, cudaMemcpy2DAsync(codes, D, src, 2 * D, D, F, k, c->stream));
    } else {
      AE_CK(c, cudaMemcpyAsync(codes, (const uint8_t*)c->w_d + (size_t)layer * D * F, D * F, k, c->stream));
    }
  }
  if (scale != nullptr)
    AE_CK(c, cudaMemcpyAsync(scale, c->fp8_tensor_scale + layer * 7 + which, sizeof(float), cudaMemcpyDeviceToHost,
                             c->stream));
  AE_CK(c, cudaStreamSynchronize(c->stream));
  return AE_OK;
}

ae_status ae_get_info(const ae_ctx* c, ae_info* info) {
  if (c == nullptr || info == nullptr) return AE_ERR_INVALID_ARG;
  info->launches_last_sample = c->launches_sample;
  info->launches_last_bind = c->launches_bind;
  info->device_bytes = c->device_bytes;
  info->sm_count = c->sm_count;
  info->path = c->d.dtype == AE_DTYPE_BF16 ? 1 : 0;
  return AE_OK;
}

}  // extern "C"
