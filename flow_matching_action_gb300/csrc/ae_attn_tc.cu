// Split-KV attention of the action rows on the tensor cores (bf16 path).
//
// The query heads of a KV group share one KV head (MQA/GQA, LoongForge Pi0.5
// blog section 3), so the (Hq / Hkv) x H action queries of a request's group
// are folded into one tall matrix, row r = head-in-group * H + token, and every
// K/V block is loaded once for all of them.
// The key set of request b is its VALID prefix rows (gathered through the bind
// table: masked and padded rows are never read) followed by its H action rows
// (actions see every valid prefix token and each other).
//
// A CTA owns (request, 128-row query tile, range of 64-key chunks) and walks
// its chunks with an online softmax:
//   S = Q K^T      tcgen05, M = 128 query rows, N = 64 keys, K = dh; S in TMEM
//   P = exp(S - m) fp32 per query row (one thread per row), bf16 into smem
//   O += P V       tcgen05, M = 128, N = dh, K = 64 keys; O stays in TMEM
// The exponent reference m is raised (and O, l rescaled in place) only when a
// chunk's maximum exceeds it by more than 8, so P <= e^8 and most chunks skip
// the rescale.  Each CTA writes its unnormalized O with (m, l); a combine
// kernel merges the ranges of a row in range order (deterministic) and
// writes the bf16 attention output o[token][head * dh + d].
#include <math.h>

#include "ae_internal.h"
#include "ae_tc.cuh"

namespace ae {
namespace {

using namespace tc;

constexpr int kAttnThreads = 128;
constexpr int kChunk = 64;            // keys per chunk
constexpr float kRescaleMargin = 8.f; // raise the exponent reference only past this

struct AttnSmem {
  uint32_t q, k[2], v[2], p, bars, total;  // byte offsets from the 1024-aligned base
};

// Q: [dh/64][128 rows][128 B] K-major.  K: [dh/64][64 keys][128 B] K-major.
// V: row-major rows of the chunk as an MN-major operand (MN = dh, K = keys):
// 1024-byte atoms of 8 keys x 64 dims, dims-atoms 1024 B apart, key-atoms
// dh/64 * 1024 B apart.  P: [128 rows][128 B] K-major.  K and V are double
// buffered so the next chunk's gathers overlap this chunk's MMAs.
__host__ __device__ inline AttnSmem attn_smem_layout(int dh) {
  AttnSmem L;
  const uint32_t kv = (uint32_t)dh * kChunk * 2;
  L.q = 0;
  L.k[0] = L.q + (uint32_t)dh * 128 * 2;
  L.k[1] = L.k[0] + kv;
  L.v[0] = L.k[1] + kv;
  L.v[1] = L.v[0] + kv;
  L.p = L.v[1] + kv;
  L.bars = L.p + 128 * kChunk * 2;
  L.total = L.bars + 64;
  return L;
}

__host__ __device__ inline uint32_t attn_tmem_cols(int dh) {
  uint32_t c = 32;
  while (c < (uint32_t)(dh + kChunk)) c <<= 1;
  return c;
}

__global__ void __launch_bounds__(kAttnThreads, 1) k_attn_tc(const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int dh = a.dh;
  const AttnSmem L = attn_smem_layout(dh);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* bar_o = bar_s + 1;
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(bar_s + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_p + 1);

  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int u = blockIdx.x;
  const int sp = u % a.max_splits;
  u /= a.max_splits;
  const int qt = u % a.q_tiles;
  u /= a.q_tiles;
  const int g = u % a.Hkv;
  const int b = u / a.Hkv;
  const int G = a.Hq / a.Hkv;  // query heads per KV head
  const int n_pre = a.n_valid[b];
  const int n_keys = n_pre + a.H;
  const int n_chunks = (n_keys + kChunk - 1) / kChunk;
  const int c_begin = sp * a.chunks_per_cta;
  const int c_end = min(c_begin + a.chunks_per_cta, n_chunks);
  if (c_begin >= c_end) return;  // uniform for the CTA
  const int n_my = c_end - c_begin;
  const int rows = G * a.H;
  const int qkvdim = (a.Hq + 2 * a.Hkv) * dh;
  const int kvdim = a.Hkv * dh;
  const int kdb = dh / 64;
  const int cpr = dh / 8;  // 16-byte chunks per head row
  const uint32_t tcols = attn_tmem_cols(dh);
  const uint32_t v_sbo = (uint32_t)kdb * 1024;

  if (threadIdx.x == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_base_p, tcols);
    tmem_relinquish();
  }

  // gathers of one chunk's K and V rows of KV head g into buffer `buf`
  auto load_chunk = [&](int c, int buf) {
    const int key0 = c * kChunk;
    const int nk = min(kChunk, n_keys - key0);
    uint8_t* ks = smem + L.k[buf];
    uint8_t* vs = smem + L.v[buf];
    for (int i = threadIdx.x; i < kChunk * cpr; i += kAttnThreads) {
      const int j = i / cpr, ch = i % cpr;
      const bf16* ksrc = a.qkv;  // any valid address when zero-filling
      const bf16* vsrc = a.qkv;
      uint32_t bytes = 0;
      if (j < nk) {
        const int key = key0 + j;
        if (key < n_pre) {
          const int prow = a.valid_idx[(size_t)b * a.max_rows + key];
          if (prow >= 0 && prow < a.total_rows) {
            ksrc = a.pk + (size_t)prow * kvdim + g * dh + ch * 8;
            vsrc = a.pv + (size_t)prow * kvdim + g * dh + ch * 8;
            bytes = 16;
          } else {
            report(a.status, kDevBounds);
          }
        } else {
          const bf16* base = a.qkv + (size_t)(b * a.H + (key - n_pre)) * qkvdim;
          ksrc = base + (a.Hq + g) * dh + ch * 8;
          vsrc = base + (a.Hq + a.Hkv + g) * dh + ch * 8;
          bytes = 16;
        }
      }
      const int grp = ch >> 3, cc = ch & 7;
      cp_async16(ks + grp * kChunk * 128 + sw128_offset(j, cc), ksrc, bytes);
      cp_async16(vs + (j >> 3) * v_sbo + grp * 1024 + sw128_offset(j & 7, cc), vsrc, bytes);
    }
  };

  // ---- Q tile (once): folded row r = 128 qt + row  ->  (head, token); then chunk 0
  for (int i = threadIdx.x; i < 128 * cpr; i += kAttnThreads) {
    const int row = i / cpr, ch = i % cpr;
    const int r = qt * 128 + row;
    const bf16* src = a.qkv;
    uint32_t bytes = 0;
    if (r < rows) {
      const int h = g * G + r / a.H, tok = r % a.H;
      src = a.qkv + (size_t)(b * a.H + tok) * qkvdim + h * dh + ch * 8;
      bytes = 16;
    }
    cp_async16(smem + L.q + (ch >> 3) * 128 * 128 + sw128_offset(row, ch & 7), src, bytes);
  }
  load_chunk(c_begin, 0);
  cp_async_commit();

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_p;
  const uint32_t tm_o = tmem, tm_s = tmem + (uint32_t)dh;
  const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
  const int row = threadIdx.x;
  float m_ref = -INFINITY, l = 0.f;
  bool failed = false;

  for (int ci = 0; ci < n_my; ++ci) {
    const int c = c_begin + ci;
    const int buf = ci & 1;
    const int nk = min(kChunk, n_keys - c * kChunk);
    // prefetch the next chunk into the other buffer (its last reader, the
    // previous chunk's P V, completed before this iteration began)
    if (ci + 1 < n_my) {
      load_chunk(c + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- S = Q K^T
    if (threadIdx.x == 0) {
      const uint32_t idesc = idesc_bf16(128, kChunk);
      for (int kb = 0; kb < kdb; ++kb) {
        const uint64_t ad = sdesc_sw128(smem_u32(smem + L.q + kb * 128 * 128));
        const uint64_t bd = sdesc_sw128(smem_u32(smem + L.k[buf] + kb * kChunk * 128));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tm_s, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(bar_s);
    }
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar_s, (uint32_t)ci & 1u, abort_flag, a.status) ? 1 : 0;
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();
    float s[kChunk];
#pragma unroll
    for (int c0 = 0; c0 < kChunk; c0 += 16) {
      float v[16];
      tmem_ld16(tm_s + lane_off + (uint32_t)c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) s[c0 + j] = v[j] * a.scale;
    }
    float cmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < kChunk; ++j)
      if (j < nk) cmax = fmaxf(cmax, s[j]);
    // raise the exponent reference; O (in TMEM) and l follow it
    float factor = 1.f;
    if (ci == 0) {
      m_ref = cmax;
    } else if (cmax > m_ref + kRescaleMargin) {
      factor = __expf(m_ref - cmax);
      m_ref = cmax;
    }
    if (__any_sync(0xffffffffu, factor != 1.f)) {
      l *= factor;
      for (int c0 = 0; c0 < dh; c0 += 16) {
        float v[16];
        tmem_ld16(tm_o + lane_off + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] *= factor;
        tmem_st16(tm_o + lane_off + (uint32_t)c0, v);
      }
    }
    uint32_t pk[kChunk / 2];
#pragma unroll
    for (int j = 0; j < kChunk; j += 2) {
      const float p0 = (j < nk) ? __expf(s[j] - m_ref) : 0.f;
      const float p1 = (j + 1 < nk) ? __expf(s[j + 1] - m_ref) : 0.f;
      const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
      // the row sum uses the bf16-rounded weights, the values P V multiplies
      const float2 pr = __bfloat1622float2(pb);
      l += pr.x + pr.y;
      pk[j / 2] = *reinterpret_cast<const uint32_t*>(&pb);
    }
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
      *reinterpret_cast<uint4*>(smem + L.p + sw128_offset(row, cc)) =
          make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- O += P V   (V as the MN-major operand: 16 keys = two 8-key atoms per step)
    if (threadIdx.x == 0) {
      const uint32_t idesc = idesc_bf16(128, dh, true);
      const uint64_t ad = sdesc_sw128(smem_u32(smem + L.p));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t bd = sdesc_sw128_mn(smem_u32(smem + L.v[buf] + k * 2 * v_sbo), 1024, v_sbo);
        mma_bf16(tm_o, ad + 2 * k, bd, idesc, (ci > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(bar_o);
    }
    ok = 1;
    if (lane == 0) ok = mbar_wait(bar_o, (uint32_t)ci & 1u, abort_flag, a.status) ? 1 : 0;
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();
  }
  cp_async_wait<0>();
  if (!failed) {
    const int r = qt * 128 + row;
    const size_t unit = ((size_t)((b * a.Hkv + g) * a.q_tiles + qt)) * a.max_splits + sp;
    float* po = a.part_o + (unit * 128 + row) * dh;
    for (int c0 = 0; c0 < dh; c0 += 16) {
      float v[16];
      tmem_ld16(tm_o + lane_off + (uint32_t)c0, v);
      if (r < rows) {
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4*>(po + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
    if (r < rows) a.part_ml[unit * 128 + row] = make_float2(m_ref, l);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// Merge the chunk ranges of every folded query row in range order; write bf16
// o[token][head * dh + d].  Block = one (folded row of a group, request), dh threads.
__global__ void k_attn_combine(const AttnArgs a, bf16* __restrict__ o) {
  pdl_trigger();
  pdl_wait();
  const int G = a.Hq / a.Hkv;
  const int g = blockIdx.x / (G * a.H), r = blockIdx.x % (G * a.H), b = blockIdx.y;
  const int qt = r / 128, row = r % 128;
  const int n_chunks = (a.n_valid[b] + a.H + kChunk - 1) / kChunk;
  const int n_splits = (n_chunks + a.chunks_per_cta - 1) / a.chunks_per_cta;
  const int d = threadIdx.x;
  const size_t unit0 = ((size_t)((b * a.Hkv + g) * a.q_tiles + qt)) * a.max_splits;
  float m = -INFINITY;
  for (int sp = 0; sp < n_splits; ++sp) m = fmaxf(m, a.part_ml[(unit0 + sp) * 128 + row].x);
  float l = 0.f, acc = 0.f;
  for (int sp = 0; sp < n_splits; ++sp) {
    const float2 ml = a.part_ml[(unit0 + sp) * 128 + row];
    const float w = __expf(ml.x - m);
    l += ml.y * w;
    acc += a.part_o[((unit0 + sp) * 128 + row) * a.dh + d] * w;
  }
  const int h = g * G + r / a.H, tok = r % a.H;
  o[(size_t)(b * a.H + tok) * (a.Hq * a.dh) + h * a.dh + d] = __float2bfloat16_rn(acc / l);
}

}  // namespace

size_t attn_smem_bytes(int dh) { return 1024 + attn_smem_layout(dh).total; }

// Work split: aim for about two CTAs per SM over the (upper-bound) chunk count.
void attn_plan(AttnArgs& a, int sm_count) {
  a.q_tiles = ((a.Hq / a.Hkv) * a.H + 127) / 128;
  const int max_chunks = (a.plan_rows + a.H + kChunk - 1) / kChunk;
  const long est = (long)a.batch * a.Hkv * a.q_tiles * max_chunks;
  int cpc = (int)((est + 2L * sm_count - 1) / (2L * sm_count));
  if (cpc < 1) cpc = 1;
  a.chunks_per_cta = cpc;
  a.max_splits = (max_chunks + cpc - 1) / cpc;
  // a fixed-size scratch: fewer, longer chunk ranges until the units fit
  while (a.max_units > 0 && (long)a.batch * a.Hkv * a.q_tiles * a.max_splits > a.max_units &&
         a.chunks_per_cta < max_chunks) {
    ++a.chunks_per_cta;
    a.max_splits = (max_chunks + a.chunks_per_cta - 1) / a.chunks_per_cta;
  }
}

size_t attn_plan_units(AttnArgs a, int sm_count) {
  attn_plan(a, sm_count);
  return (size_t)a.batch * a.Hkv * a.q_tiles * a.max_splits;
}

// Work units never exceed 2 * sm_count + batch * Hkv * q_tiles: a plan with one
// chunk per CTA has at most 2 * sm_count units, and rounding the split count
// up adds at most one unit per (request, KV head, query tile).
size_t attn_part_units(int max_batch, int H, int Hq, int Hkv, int max_rows, int sm_count) {
  (void)max_rows;
  const int q_tiles = ((Hq / Hkv) * H + 127) / 128;
  return (size_t)2 * sm_count + (size_t)max_batch * Hkv * q_tiles;
}

cudaError_t attn_kernel_setup() {
  return cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
}

cudaError_t launch_attn_tc(AttnArgs a, bf16* o, int sm_count, cudaStream_t s, bool pdl) {
  attn_plan(a, sm_count);
  const size_t smem = attn_smem_bytes(a.dh);
  const unsigned grid = (unsigned)(a.batch * a.Hkv * a.q_tiles * a.max_splits);
  cudaError_t e = launch_k(k_attn_tc, dim3(grid), dim3(kAttnThreads), smem, s, pdl, a);
  if (e != cudaSuccess) return e;
  return launch_k(k_attn_combine, dim3(a.Hq * a.H, a.batch), dim3(a.dh), 0, s, pdl, a, o);
}

}  // namespace ae
