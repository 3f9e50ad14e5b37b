// Split-KV attention of the action rows on the tensor cores (bf16 path).
//
// The query heads of a KV group share one KV head (MQA/GQA, LoongForge Pi0.5
// blog section 3), so the (Hq / Hkv) x H action queries of a request's group
// are folded into one tall matrix and every K/V block is loaded once for all
// of them.  Each head's H rows are padded to a multiple of 16 in the fold
// (row r = head-in-group * Hp + token, Hp = H rounded up to 16) so the query
// tile arrives as 16-row TMA boxes.
// The key set of request b is its VALID prefix rows (through the bind table:
// masked and padded rows are never read) followed by its H action rows
// (actions see every valid prefix token and each other).  A 64-key chunk whose
// rows form one contiguous run of valid prefix rows (the common case) arrives
// as TMA boxes; any other chunk is gathered row by row with cp.async.  V is
// stored exactly like K (rows of 64-dim, 128-byte-swizzled blocks) and read as
// the MN-major operand of P V.
//
// A CTA owns (request, KV head, 128-row query tile, range of chunks) and walks
// its chunks with an online softmax, the next chunk's K/V loading while the
// current one computes:
//   S = Q K^T      tcgen05, M = 128 query rows, N = 64 keys, K = dh; S in TMEM
//   P = exp(S - m) fp32 per query row (two threads per row, 32 keys each;
//                  the row's maximum and sum combined through shared memory),
//                  bf16 back into TMEM over the S columns already read
//   O += P V       tcgen05 with P as the TMEM A operand, M = 128, N = dh,
//                  K = 64 keys; O stays in TMEM
// The exponent reference m is raised (and O, l rescaled in place) only when a
// chunk's maximum exceeds it by more than 8, so P <= e^8 and most chunks skip
// the rescale.  Each CTA stores its partial (TMA store) with (m, l): bf16 rows
// of O / l by default, fp32 O where the caller supplies its own scratch; a
// combine kernel merges the ranges of a row in range
// order (deterministic) and writes the bf16 attention output
// o[token][head * dh + d].
#include <math.h>
#include <string.h>

#include <type_traits>

#include "ae_internal.h"
#include "ae_tc.cuh"

namespace ae {
namespace {

using namespace tc;

constexpr int kAttnThreads = 256;  // two warps per TMEM lane quarter
constexpr int kChunk = 64;             // keys per chunk
constexpr float kRescaleMargin = 8.f;  // raise the exponent reference only past this
constexpr int kSkip = -0x40000000;     // gather code: zero-fill

__host__ __device__ inline int fold_rows_per_head(int H) { return (H + 15) & ~15; }

// Two floats rounded to bf16 and packed (first in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

struct AttnSmem {
  uint32_t q, k[2], v[2], bars, idx, total;  // byte offsets from the 1024-aligned base
};

// Q: [dh/64][128 rows][128 B].  K and V: [dh/64][64 keys][128 B] (8 KB blocks),
// double buffered.  All 128-byte swizzled.
__host__ __device__ inline AttnSmem attn_smem_layout(int dh) {
  AttnSmem L;
  const uint32_t kv = (uint32_t)dh * kChunk * 2;
  L.q = 0;
  L.k[0] = L.q + (uint32_t)dh * 128 * 2;
  L.k[1] = L.k[0] + kv;
  L.v[0] = L.k[1] + kv;
  L.v[1] = L.v[0] + kv;
  L.bars = L.v[1] + kv;  // bar_s, bar_o, bar_q, bar_kv[2], TMEM base, abort flag
  L.idx = L.bars + 64;              // [2][kChunk] gather codes of the two K/V buffers
  L.total = L.idx + 2 * kChunk * 4 + 2 * 2 * 128 * 4;  // + per-half row maxima and sums [2][2][128]
  return L;
}

__host__ __device__ inline uint32_t attn_tmem_cols(int dh) {
  uint32_t c = 32;
  while (c < (uint32_t)(dh + kChunk)) c <<= 1;
  return c;
}

// Chunk c of KV head g into buffer `buf`, in two parts.  chunk_codes() reads
// the chunk's gather codes into shared memory (>= 0 physical prefix row,
// -1 - i action row i, kSkip zero-fill) and, when the chunk is one contiguous
// run of 64 valid prefix rows, starts its TMA loads (completion on bar_kv) and
// returns true.  Otherwise chunk_gather() copies it row by row with cp.async
// (one commit group).  Both are uniform for the CTA.  Prefix rows and codes
// come from the binding, so chunk_codes() may run before the preceding kernel
// has finished; chunk_gather() reads action rows and must run after it.
template <int DH>
__device__ __forceinline__ bool chunk_codes(const AttnArgs& a, const CUtensorMap* kmap,
                                            const CUtensorMap* vmap, uint8_t* smem, const AttnSmem& L,
                                            uint64_t* bar_kv, int b, int g, int n_pre, int n_keys,
                                            int c, int buf, bool whole_rows) {
  constexpr int kdb = DH / 64;
  const int key0 = c * kChunk;
  const int nk = min(kChunk, n_keys - key0);
  int* ix = reinterpret_cast<int*>(smem + L.idx) + buf * kChunk;
  if (threadIdx.x < kChunk) {
    const int j = threadIdx.x, key = key0 + j;
    int code = kSkip;
    if (j < nk) {
      if (key < n_pre) {
        const int prow = a.valid_idx[(size_t)b * a.max_rows + key];
        if (prow >= 0 && prow < a.total_rows) code = prow;
        else report(a.status, kDevBounds);
      } else {
        code = -1 - (key - n_pre);
      }
    }
    ix[j] = code;
  }
  __syncthreads();
  // codes increase strictly over a chunk's prefix keys: first and last decide
  const bool contiguous = nk == kChunk && ix[0] >= 0 && ix[kChunk - 1] - ix[0] == kChunk - 1;
  if (contiguous && threadIdx.x == 0) {
    uint8_t* ks = smem + L.k[buf];
    uint8_t* vs = smem + L.v[buf];
    mbar_arrive_expect_tx(&bar_kv[buf], 2u * kdb * kChunk * 128);
    const int row = a.layer_row0 + ix[0];
    if (whole_rows) {
      // K and V as one box each (the maps' 3-D views: 64 rows x DH columns land
      // as DH / 64 swizzled [64 rows][128 B] blocks): two TMA issues, not 2 DH / 64
      tma_load_3d_nohint(ks, kmap, &bar_kv[buf], 0, row, g * kdb);
      tma_load_3d_nohint(vs, vmap, &bar_kv[buf], 0, row, g * kdb);
    } else {
#pragma unroll
      for (int kb = 0; kb < kdb; ++kb) {
        tma_load_2d_nohint(ks + kb * kChunk * 128, kmap, &bar_kv[buf], g * DH + kb * 64, row);
        tma_load_2d_nohint(vs + kb * kChunk * 128, vmap, &bar_kv[buf], g * DH + kb * 64, row);
      }
    }
  }
  return contiguous;
}

template <int DH>
__device__ __forceinline__ void chunk_gather(const AttnArgs& a, uint8_t* smem, const AttnSmem& L,
                                             int b, int g, int buf) {
  constexpr int CPR = DH / 8;                    // 16-byte pieces per row
  constexpr int RPW = CPR >= 32 ? 1 : 32 / CPR;  // rows per warp instruction
  constexpr int PPL = CPR >= 32 ? CPR / 32 : 1;  // pieces per lane per row
  const int* ix = reinterpret_cast<const int*>(smem + L.idx) + buf * kChunk;
  uint8_t* ks = smem + L.k[buf];
  uint8_t* vs = smem + L.v[buf];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / (32 / RPW);  // row within this warp instruction
  const int pl = lane % (32 / RPW);   // piece index of the lane
  const int kvdim = a.Hkv * DH, qkvdim = (a.Hq + 2 * a.Hkv) * DH;
  for (int j0 = warp * RPW; j0 < kChunk; j0 += (kAttnThreads / 32) * RPW) {
    const int j = j0 + sub;
    const int code = ix[j];
    const bf16* kr = a.qkv;  // any valid address when zero-filling
    const bf16* vr = a.qkv;
    uint32_t bytes = 0;
    if (code >= 0) {
      kr = a.pk + (size_t)code * kvdim + g * DH;
      vr = a.pv + (size_t)code * kvdim + g * DH;
      bytes = 16;
    } else if (code != kSkip) {
      const bf16* base = a.qkv + (size_t)(b * a.H + (-1 - code)) * qkvdim;
      kr = base + (a.Hq + g) * DH;
      vr = base + (a.Hq + a.Hkv + g) * DH;
      bytes = 16;
    }
#pragma unroll
    for (int e = 0; e < PPL; ++e) {
      const int ch = pl + e * 32;
      const uint32_t off = (ch >> 3) * kChunk * 128 + sw128_offset(j, ch & 7);
      cp_async16(ks + off, bytes ? kr + ch * 8 : kr, bytes);
      cp_async16(vs + off, bytes ? vr + ch * 8 : vr, bytes);
    }
  }
  cp_async_commit();
}

template <int DH>
__device__ __forceinline__ bool load_kv_chunk(const AttnArgs& a, const CUtensorMap* kmap,
                                              const CUtensorMap* vmap, uint8_t* smem,
                                              const AttnSmem& L, uint64_t* bar_kv, int b, int g,
                                              int n_pre, int n_keys, int c, int buf) {
  const bool tma = chunk_codes<DH>(a, kmap, vmap, smem, L, bar_kv, b, g, n_pre, n_keys, c, buf, true);
  if (!tma) chunk_gather<DH>(a, smem, L, b, g, buf);
  return tma;
}

// O16: partials stored as bf16 rows of O / l (else fp32 O); one instantiation
// each, so a launch carries only the store it runs.
template <int DH, bool O16>
__global__ void __launch_bounds__(kAttnThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap kmap3,
              const __grid_constant__ CUtensorMap vmap3, const __grid_constant__ CUtensorMap omap,
              const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // keeps the shared address space
  constexpr int dh = DH;
  constexpr int kdb = dh / 64;
  const AttnSmem L = attn_smem_layout(dh);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* bar_o = bar_s + 1;
  uint64_t* bar_q = bar_s + 2;
  uint64_t* bar_kv = bar_s + 3;  // [2]
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(bar_s + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_p + 1);

  // Everything up to the first chunk's prefix loads depends only on the
  // binding (n_valid, valid_idx, prefix K/V) and may overlap the preceding
  // kernel; the query tile and action rows are read after pdl_wait().
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int u = blockIdx.x;
  const int sp = u % a.max_splits;
  u /= a.max_splits;
  const int qt = u % a.q_tiles;
  u /= a.q_tiles;
  const int g = u % a.Hkv;
  const int b = u / a.Hkv;
  const int G = a.Hq / a.Hkv;  // query heads per KV head
  const int Hp = fold_rows_per_head(a.H);
  const int n_pre = a.n_valid[b];
  const int n_keys = n_pre + a.H;
  const int n_chunks = (n_keys + kChunk - 1) / kChunk;
  const int c_begin = sp * a.chunks_per_cta;
  const int c_end = min(c_begin + a.chunks_per_cta, n_chunks);
  if (c_begin >= c_end) {  // uniform for the CTA
    pdl_wait();
    return;
  }
  const int n_my = c_end - c_begin;
  const uint32_t tcols = attn_tmem_cols(dh);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bar_s[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&kmap3);
    prefetch_tensormap(&vmap3);
  }
  if (warp == 0) {
    tmem_alloc(tmem_base_p, tcols);
    tmem_relinquish();
  }
  __syncthreads();
  // the first chunk loads while the preceding kernel finishes: boxes of 64
  // columns; chunks inside the loop use the whole-row boxes (fewer issues on
  // the critical path)
  bool tma_cur = chunk_codes<DH>(a, &kmap, &vmap, smem, L, bar_kv, b, g, n_pre, n_keys, c_begin, 0, false);
  // bit i: buffer i has a TMA copy in flight (thread 0's view; drained on
  // the way out after a failure)
  uint32_t kv_pending = tma_cur ? 1u : 0u;
  pdl_wait();
  if (!tma_cur) chunk_gather<DH>(a, smem, L, b, g, 0);
  // ---- Q tile by TMA: groups of a.q_box rows of the fold (q_box divides the
  //      padded head length, so a group never straddles heads)
  if (threadIdx.x == 0) {
    const int QB = a.q_box, n_rg = 128 / QB;
    int nbox = 0;
    for (int rg = 0; rg < n_rg; ++rg)
      if ((qt * 128 + rg * QB) / Hp < G) ++nbox;
    mbar_arrive_expect_tx(bar_q, (uint32_t)nbox * kdb * QB * 128);
    for (int rg = 0; rg < n_rg; ++rg) {
      const int r0 = qt * 128 + rg * QB;
      const int hh = r0 / Hp;
      if (hh >= G) continue;
      const int tok0 = r0 - hh * Hp;
      const int col = (g * G + hh) * dh;
#pragma unroll
      for (int kb = 0; kb < kdb; ++kb)
        tma_load_2d_nohint(smem + L.q + kb * 128 * 128 + rg * QB * 128, &qmap, bar_q, col + kb * 64,
                           b * a.H + tok0);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_p;
  const uint32_t tm_o = tmem, tm_s = tmem + (uint32_t)dh;
  // the two warps of a TMEM lane quarter take the same 32 rows; half h takes
  // keys 32 h.. of a chunk and the O columns of its half
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
  const int row = threadIdx.x & 127;
  const int half = threadIdx.x >> 7;
  float* red_m = reinterpret_cast<float*>(smem + L.idx + 2 * kChunk * 4);  // [2][128]
  float* red_l = red_m + 2 * 128;                                         // [2][128]
  float m_ref = -INFINITY, l = 0.f;
  bool failed = false;
  int fail_at = 0;                  // 1: S = Q K^T in flight, 2: P V in flight
  uint32_t fail_par = 0u;           // parity of that MMA's commit
  uint32_t kv_phase = 0u;           // bit i: parity of buffer i's next load (thread 0)
  bool q_pending = true;

  for (int ci = 0; ci < n_my; ++ci) {
    const int c = c_begin + ci;
    const int buf = ci & 1;
    const int nk = min(kChunk, n_keys - c * kChunk);
    const bool has_next = ci + 1 < n_my;
    int ok = 1;
    if (!tma_cur) {
      cp_async_wait<0>();  // the next chunk's copies start only after S is issued
      fence_proxy_async_smem();
    } else if (threadIdx.x == 0) {
      ok = mbar_wait(&bar_kv[buf], (kv_phase >> buf) & 1u, abort_flag, a.status) ? 1 : 0;
      if (ok) {
        kv_phase ^= 1u << buf;
        kv_pending &= ~(1u << buf);
      }
    }
    if (ci == 0 && threadIdx.x == 0 && ok) {
      ok = mbar_wait(bar_q, 0, abort_flag, a.status) ? 1 : 0;
      if (ok) q_pending = false;
    }
    tc_fence_before();
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();
    // ---- S = Q K^T
    if (threadIdx.x == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, kChunk);
#pragma unroll
      for (int kb = 0; kb < kdb; ++kb) {
        const uint64_t ad = sdesc_sw128(smem_u32(smem + L.q + kb * 128 * 128));
        const uint64_t bd = sdesc_sw128(smem_u32(smem + L.k[buf] + kb * kChunk * 128));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tm_s, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(bar_s);
    }
    // the next chunk starts loading into the other buffer while S runs: its
    // last readers, the previous chunk's S and P V, have completed (their
    // waits came before this point), and neither the gather codes' global
    // reads nor the copies' issue sit between P V and this chunk's S
    bool tma_next = false;
    if (has_next) {
      tma_next = load_kv_chunk<DH>(a, &kmap3, &vmap3, smem, L, bar_kv, b, g, n_pre, n_keys, c + 1, buf ^ 1);
      if (tma_next) kv_pending |= 1u << (buf ^ 1);
    }
    ok = 1;
    if (lane == 0) ok = mbar_wait(bar_s, (uint32_t)ci & 1u, abort_flag, a.status) ? 1 : 0;
    if (__syncthreads_or(!ok)) {
      failed = true;
      fail_at = 1;
      fail_par = (uint32_t)ci & 1u;
      break;
    }
    tc_fence_after();
    // scores in the log2 domain: s * scale * log2(e), so exp() becomes one exp2
    const float sl2 = a.scale * 1.4426950408889634f;
    float s[32];
    tmem_ld32(tm_s + lane_off + (uint32_t)(32 * half), s);
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      s[j] *= sl2;
      if (32 * half + j < nk) mx[j & 3] = fmaxf(mx[j & 3], s[j]);
    }
    red_m[half * 128 + row] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    __syncthreads();
    const float cmax = fmaxf(red_m[row], red_m[128 + row]);
    // raise the exponent reference; O (in TMEM) and l follow it
    float factor = 1.f;
    if (ci == 0) {
      m_ref = cmax;
    } else if (cmax > m_ref + kRescaleMargin * 1.4426950408889634f) {
      factor = ex2_fast(m_ref - cmax);
      m_ref = cmax;
    }
    if (__any_sync(0xffffffffu, factor != 1.f)) {
      l *= factor;
#pragma unroll 1
      for (int c0 = half * (dh / 2); c0 < (half + 1) * (dh / 2); c0 += 16) {
        float v[16];
        tmem_ld16(tm_o + lane_off + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] *= factor;
        tmem_st16(tm_o + lane_off + (uint32_t)c0, v);
      }
    }
    uint32_t pk[16];
    float ls[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains, added in a fixed order
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const int key = 32 * half + j;
      const float p0 = (key < nk) ? ex2_fast(s[j] - m_ref) : 0.f;
      const float p1 = (key + 1 < nk) ? ex2_fast(s[j + 1] - m_ref) : 0.f;
      const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
      // the row sum uses the bf16-rounded weights, the values P V multiplies
      const float2 pr = __bfloat1622float2(pb);
      ls[(j >> 1) & 3] += pr.x + pr.y;
      pk[j / 2] = *reinterpret_cast<const uint32_t*>(&pb);
    }
    red_l[half * 128 + row] = (ls[0] + ls[1]) + (ls[2] + ls[3]);
    {
      // P over the S columns already read (every thread loaded its S before
      // the maximum exchange): column j of the row holds keys 2j, 2j + 1, the
      // A operand of P V in tensor memory
      float pf[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) pf[j] = __uint_as_float(pk[j]);
      tmem_st16(tm_s + lane_off + (uint32_t)(16 * half), pf);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    l += red_l[row] + red_l[128 + row];
    // ---- O += P V: P from TMEM (8 columns per 16 keys); V rows are the
    //      MN-major operand (dims along MN in 64-dim blocks 8 KB apart, keys
    //      along K in 8-key atoms 1 KB apart)
    if (threadIdx.x == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, dh, true);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t bd = sdesc_sw128_mn(smem_u32(smem + L.v[buf] + k * 2048), kChunk * 128, 1024);
        mma_bf16_ts(tm_o, tm_s + (uint32_t)(8 * k), bd, idesc, (ci > 0 || k > 0) ? 1u : 0u);
      }
      mma_commit(bar_o);
    }
    ok = 1;
    if (lane == 0) ok = mbar_wait(bar_o, (uint32_t)ci & 1u, abort_flag, a.status) ? 1 : 0;
    if (__syncthreads_or(!ok)) {
      failed = true;
      fail_at = 2;
      fail_par = (uint32_t)ci & 1u;
      break;
    }
    tc_fence_after();
    tma_cur = tma_next;
  }
  cp_async_wait<0>();
  if (failed && threadIdx.x == 0) {
    // no TMA copy may still be writing shared memory, nor an MMA tensor
    // memory, when the CTA exits: bounded waits that hold after an abort
    if (q_pending) mbar_drain(bar_q, 0, a.status);
    for (int i = 0; i < 2; ++i)
      if ((kv_pending >> i) & 1u) mbar_drain(&bar_kv[i], (kv_phase >> i) & 1u, a.status);
    if (fail_at == 1) mbar_drain(bar_s, fail_par, a.status);
    if (fail_at == 2) mbar_drain(bar_o, fail_par, a.status);
  }
  __syncthreads();  // every chunk buffer is free: reuse K/V space to stage O
  if (!failed) {
    // O rows -> 128-byte-swizzled staging boxes (the K/V buffers hold exactly
    // 128 x dh floats), then TMA stores
    const int r = qt * 128 + row;
    const bool valid_row = r / Hp < G && r % Hp < a.H;
    const size_t unit = ((size_t)((b * a.Hkv + g) * a.q_tiles + qt)) * a.max_splits + sp;
    uint8_t* stg = smem + L.k[0];
    if constexpr (O16) {
      // bf16 rows of O / l (half the bytes of fp32 partials): boxes of 64
      // columns, each stored by its half's first thread as soon as the half's
      // four warps have staged it (the store overlaps the next box's staging)
      const float inv_l = 1.f / l;
#pragma unroll 1
      for (int c0 = 64 * half; c0 < dh; c0 += 128) {
        float v[64];
        tmem_ld64(tm_o + lane_off + (uint32_t)c0, v);
        uint8_t* box = stg + (c0 >> 6) * (128 * 128);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<uint4*>(box + sw128_offset(row, q)) =
              make_uint4(pack_bf16x2(v[8 * q] * inv_l, v[8 * q + 1] * inv_l),
                         pack_bf16x2(v[8 * q + 2] * inv_l, v[8 * q + 3] * inv_l),
                         pack_bf16x2(v[8 * q + 4] * inv_l, v[8 * q + 5] * inv_l),
                         pack_bf16x2(v[8 * q + 6] * inv_l, v[8 * q + 7] * inv_l));
        fence_proxy_async_smem();
        if (half == 0) asm volatile("bar.sync 1, 128;" ::: "memory");
        else asm volatile("bar.sync 2, 128;" ::: "memory");
        if (row == 0) tma_store_2d(&omap, box, c0, (int)(unit * 128));
      }
      if (row == 0) bulk_commit();
    } else {
#pragma unroll 1
      for (int c0 = 64 * half; c0 < dh; c0 += 128) {
        float v[64];
        tmem_ld64(tm_o + lane_off + (uint32_t)c0, v);
#pragma unroll
        for (int q = 0; q < 16; ++q) {  // 16 float4 = two 32-column boxes
          const int col = c0 + 4 * q;
          uint8_t* box = stg + (col >> 5) * (128 * 128);
          *reinterpret_cast<float4*>(box + sw128_offset(row, (col & 31) >> 2)) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
    }
    // the stored maximum is in the log2 domain of the scaled scores
    if (valid_row && half == 0) a.part_ml[unit * 128 + row] = make_float2(m_ref, l);
    if constexpr (O16) {
      if (row == 0) bulk_wait_read_all();  // this half's stores have read the staging
    } else {
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        for (int bx = 0; bx < dh / 32; ++bx) tma_store_2d(&omap, stg + bx * (128 * 128), bx * 32, (int)(unit * 128));
        bulk_commit();
        bulk_wait_read_all();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// Merge the chunk ranges of every query row in range order; write bf16
// o[token][head * dh + d].  One warp per (head, token) row, 8 rows per block;
// lane l merges dims 8l.. (16-byte loads and stores), all ranges' loads issued
// together, merged with an online rescale (deterministic order).
constexpr int kCombineRows = 8;

template <bool O16>
__global__ void __launch_bounds__(32 * kCombineRows) k_attn_combine(const AttnArgs a, bf16* __restrict__ o) {
  pdl_trigger();
  pdl_wait();
  const int G = a.Hq / a.Hkv;
  const int Hp = fold_rows_per_head(a.H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ri = blockIdx.x * kCombineRows + warp;  // row over (request, KV head, head in group, token)
  if (ri >= a.batch * a.Hq * a.H) return;
  const int per_b = a.Hq * a.H;
  const int b = ri / per_b, hr0 = ri - b * per_b;
  const int g = hr0 / (G * a.H), hr = hr0 - g * (G * a.H);
  const int hh = hr / a.H, tok = hr - hh * a.H;
  const int r = hh * Hp + tok;  // folded row
  const int qt = r / 128, row = r % 128;
  const int n_chunks = (a.n_valid[b] + a.H + kChunk - 1) / kChunk;
  const int n_splits = (n_chunks + a.chunks_per_cta - 1) / a.chunks_per_cta;
  const size_t unit0 = ((size_t)((b * a.Hkv + g) * a.q_tiles + qt)) * a.max_splits;
  bf16* orow = o + (size_t)(b * a.H + tok) * (a.Hq * a.dh) + (g * G + hh) * a.dh;
  for (int d0 = 8 * lane; d0 < a.dh; d0 += 256) {
    float m = -INFINITY, l = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < n_splits; s0 += 8) {
      float2 ml[8];
      float pv[8][8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool in = s0 + j < n_splits;
        const size_t rw = (unit0 + s0 + j) * 128 + row;
        ml[j] = in ? __ldcg(a.part_ml + rw) : make_float2(-INFINITY, 0.f);
        if constexpr (O16) {  // rows of O / l: weight l back in below
          const uint4 q = in ? __ldcg(reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(a.part_o) +
                                                                      rw * a.dh + d0))
                             : make_uint4(0u, 0u, 0u, 0u);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            pv[j][2 * i] = f.x;
            pv[j][2 * i + 1] = f.y;
          }
        } else {
          const float4* src = reinterpret_cast<const float4*>(a.part_o + rw * a.dh + d0);
          const float4 x0 = in ? __ldcg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 x1 = in ? __ldcg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
          pv[j][0] = x0.x; pv[j][1] = x0.y; pv[j][2] = x0.z; pv[j][3] = x0.w;
          pv[j][4] = x1.x; pv[j][5] = x1.y; pv[j][6] = x1.z; pv[j][7] = x1.w;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (s0 + j >= n_splits) break;
        const float mn = fmaxf(m, ml[j].x);
        const float ra = ex2_fast(m - mn), rb = ex2_fast(ml[j].x - mn);
        const float wv = O16 ? ml[j].y * rb : rb;  // weight of this range's values
        l = l * ra + ml[j].y * rb;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = acc[i] * ra + pv[j][i] * wv;
        m = mn;
      }
    }
    const float il = 1.f / l;
    *reinterpret_cast<uint4*>(orow + d0) =
        make_uint4(pack_bf16x2(acc[0] * il, acc[1] * il), pack_bf16x2(acc[2] * il, acc[3] * il),
                   pack_bf16x2(acc[4] * il, acc[5] * il), pack_bf16x2(acc[6] * il, acc[7] * il));
  }
}

}  // namespace

size_t attn_smem_bytes(int dh) { return 1024 + attn_smem_layout(dh).total; }

// Work split: aim for about two CTAs per SM over the (upper-bound) chunk count.
void attn_plan(AttnArgs& a, int sm_count) {
  a.q_tiles = ((a.Hq / a.Hkv) * fold_rows_per_head(a.H) + 127) / 128;
  const int max_chunks = (a.plan_rows + a.H + kChunk - 1) / kChunk;
  int cpc = 1;
  if (a.host_lens != nullptr) {
    // Chunk range per CTA that minimizes the makespan of whole waves of one
    // CTA per SM, a CTA costing its chunks plus about two chunks of prologue
    // and partial store (fit to GB300 measurements at batch 16), over the
    // bound requests' physical lengths; ties keep the shorter range.
    long best = -1;
    for (int c = 1; c <= max_chunks; ++c) {
      long ctas = 0;
      for (int b = 0; b < a.batch; ++b) {
        const int ch = (a.host_lens[b] + a.H + kChunk - 1) / kChunk;
        ctas += (long)a.Hkv * a.q_tiles * ((ch + c - 1) / c);
      }
      const long cost = ((ctas + sm_count - 1) / sm_count) * (c + 2);
      if (best < 0 || cost < best) {
        best = cost;
        cpc = c;
      }
    }
  } else {
    const long est = (long)a.batch * a.Hkv * a.q_tiles * max_chunks;
    cpc = (int)((est + 2L * sm_count - 1) / (2L * sm_count));
    if (cpc < 1) cpc = 1;
  }
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
  const int q_tiles = ((Hq / Hkv) * fold_rows_per_head(H) + 127) / 128;
  return (size_t)2 * sm_count + (size_t)max_batch * Hkv * q_tiles;
}

template <int DH>
cudaError_t attn_attrs() {
  cudaError_t e = cudaSuccess;
  for (auto kern : {k_attn_tc<DH, false>, k_attn_tc<DH, true>}) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  }
  return e;
}

cudaError_t attn_kernel_setup() {
  cudaError_t e = attn_attrs<64>();
  if (e == cudaSuccess) e = attn_attrs<128>();
  if (e == cudaSuccess) e = attn_attrs<256>();
  for (auto kern : {k_attn_combine<false>, k_attn_combine<true>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  return e;
}

static unsigned combine_blocks(const AttnArgs& a) {
  return (unsigned)((a.batch * a.Hq * a.H + kCombineRows - 1) / kCombineRows);
}

cudaError_t launch_attn_tc(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& kmap3, const CUtensorMap& vmap3, const CUtensorMap& omap_f32, const CUtensorMap* omap16, AttnArgs a, bf16* o, int sm_count,
                           cudaStream_t s, bool pdl) {
  attn_plan(a, sm_count);
  // bf16 rows of O / l halve the partials' bytes (store and combine)
  a.o16 = omap16 != nullptr ? 1 : 0;
  const CUtensorMap& omap = a.o16 ? *omap16 : omap_f32;
  const unsigned grid = (unsigned)(a.batch * a.Hkv * a.q_tiles * a.max_splits);
  const size_t smem = attn_smem_bytes(a.dh);
  auto go = [&](auto o16_tag) {
    constexpr bool O16 = decltype(o16_tag)::value;
    cudaError_t r;
    switch (a.dh) {
      case 64: r = launch_k(k_attn_tc<64, O16>, dim3(grid), dim3(kAttnThreads), smem, s, pdl, qmap, kmap, vmap, kmap3, vmap3, omap, a); break;
      case 128: r = launch_k(k_attn_tc<128, O16>, dim3(grid), dim3(kAttnThreads), smem, s, pdl, qmap, kmap, vmap, kmap3, vmap3, omap, a); break;
      default: r = launch_k(k_attn_tc<256, O16>, dim3(grid), dim3(kAttnThreads), smem, s, pdl, qmap, kmap, vmap, kmap3, vmap3, omap, a); break;
    }
    if (r != cudaSuccess) return r;
    return launch_k(k_attn_combine<O16>, dim3(combine_blocks(a)), dim3(32 * kCombineRows), 0, s, pdl, a, o);
  };
  return a.o16 ? go(std::true_type()) : go(std::false_type());
}

}  // namespace ae
