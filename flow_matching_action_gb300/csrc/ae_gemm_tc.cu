// tcgen05 GEMMs of the bf16 path and the elementwise kernels between them.
//
// Swap-AB: a CTA computes a 128-row slab of a weight matrix against a tile of
// up to 256 action tokens, D[n, t] = sum_k W[n, k] X[t, k].  The weight rows
// are the MMA's M = 128 operand and the token tile is its N operand, so a
// 50-token chunk costs a 64-wide tile instead of a 128-row one.  Both operands
// arrive by TMA into 128-byte-swizzled shared memory (weights evict-first in
// L2 when one token tile reads them: each is read once per flow step); the
// fp32 accumulator lives in TMEM.
// Merged Q/K/V and gate/up weights follow sglang PR #34599, item 1.
//
// Epilogues:
//   kEQkvRope   RoPE (rotate_half pairs) on q and k, bf16 q|k|v store
//   kEGeglu     gelu_tanh(g) * u of the interleaved gate/up rows, bf16 store
//   kEPartial   fp32 split-K partials, summed in split order later
// The kernels after the GEMMs fuse the rest of the layer (LoongForge Pi0.5
// blog, section 2): split-K sum + gated residual + the NEXT adaRMS (rms over
// the row, (1 + scale), + shift) into the bf16 operand of the next GEMM.
#include <math.h>
#include <string.h>

#include "ae_internal.h"
#include "ae_tc.cuh"

namespace ae {
namespace {

using namespace tc;

// Warp 0 issues TMA, warp 1 MMA, warps 2.. run the epilogue: EW = 4 (one per
// TMEM lane quarter) for token tiles up to 64, EW = 8 (two per quarter, each
// taking half of the token columns) for longer tiles, whose epilogue would
// otherwise be a long serial chain per thread.
constexpr int kThreadsFor(int ew) { return 64 + 32 * ew; }
constexpr int kATileBytes = 128 * 128;  // 128 weight rows x 64 bf16

// gelu_tanh(g) = 0.5 g (1 + tanh(u)), u = sqrt(2/pi) (g + 0.044715 g^3), written
// with 1 + tanh(u) = 2 / (1 + e^{-2u}): one exponential and one division.
__device__ __forceinline__ float gelu_tanh(float g) {
  const float u2 = 1.5957691216057308f * (g + 0.044715f * g * g * g);
  return __fdividef(g, 1.f + __expf(-u2));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Named barrier with a compile-time id, so the kernel reserves only the
// barriers it uses (ids 1..5) and co-resident CTAs keep theirs.
template <int ID>
__device__ __forceinline__ void named_bar(int n) {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "r"(n) : "memory");
}

__device__ __forceinline__ void quarter_bar(int q) {  // the two epilogue warps of lane quarter q
  switch (q) {
    case 0: named_bar<2>(64); break;
    case 1: named_bar<3>(64); break;
    case 2: named_bar<4>(64); break;
    default: named_bar<5>(64); break;
  }
}

template <int EW>
__global__ void __launch_bounds__(kThreadsFor(EW), 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap amap,
              const __grid_constant__ CUtensorMap omap, const __grid_constant__ TcGemmArgs a) {
  constexpr int kEpiWarps = EW;
  constexpr int kEpiThreads = 32 * EW;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int S = a.stages;
  const int btile = a.tok_tile * 128;
  uint8_t* smA = smem;
  uint8_t* smB = smA + (size_t)S * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smB + (size_t)S * btile);
  uint64_t* empty = full + S;
  uint64_t* tmem_full = empty + S;
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(tmem_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_p + 1);
  volatile int* votes = reinterpret_cast<volatile int*>(tmem_base_p + 2);  // [kEpiWarps]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int idx = blockIdx.x;
  const int n_tile = idx % a.n_tiles;
  idx /= a.n_tiles;
  const int tt = idx % a.tok_tiles;
  const int ks = idx / a.tok_tiles;
  const int kb_begin = (int)((long)ks * a.kb_total / a.ksplit);
  const int kb_end = (int)((long)(ks + 1) * a.kb_total / a.ksplit);
  const int n_it = kb_end - kb_begin;
  const int t0 = tt * a.tok_tile;
  auto kcol = [&](int it) { return (kb_begin + it) * 64; };
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  const uint32_t tmem_cols = a.tmem_cols;
  if (warp == 1) {
    tmem_alloc(tmem_base_p, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_base_p;

  if (warp == 0) {
    // ---------------- TMA producer: weight slab + token tile per 64-wide K block
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&amap);
      // a weight slab read by one token tile is not read again this flow step:
      // evict it first; with several token tiles the other tiles' CTAs read it
      // moments later, so it keeps the normal policy
      const uint64_t pol_w = a.tok_tiles > 1 ? policy_evict_normal() : policy_evict_first();
      const int row = a.w_row0 + n_tile * 128;
      const uint32_t bytes = kATileBytes + (uint32_t)btile;
      // Weights do not depend on the previous kernel: fill the first stages and
      // start pulling this slab of the next layer into L2 before waiting on it.
      const int pre = n_it < S ? n_it : S;
      for (int it = 0; it < pre; ++it) {
        mbar_arrive_expect_tx(&full[it], bytes);
        tma_load_2d(smA + (size_t)it * kATileBytes, &wmap, &full[it], kcol(it), row, pol_w);
      }
      if (a.w_next_row0 >= 0)
        for (int it = 0; it < n_it; ++it)
          tma_prefetch_l2_2d(&wmap, (kb_begin + it) * 64, a.w_next_row0 + n_tile * 128);
      pdl_wait();
      for (int it = 0; it < pre; ++it)
        tma_load_2d_nohint(smB + (size_t)it * btile, &amap, &full[it], kcol(it), t0);
      int it = pre;
      for (; it < n_it; ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, a.status)) break;
        const int kc = kcol(it);
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_2d(smA + (size_t)s * kATileBytes, &wmap, &full[s], kc, row, pol_w);
        tma_load_2d_nohint(smB + (size_t)s * btile, &amap, &full[s], kc, t0);
      }
      // drain: no copy may still be in flight when the CTA exits
      for (int j = it - S > 0 ? it - S : 0; j < it; ++j)
        mbar_wait(&full[j % S], (uint32_t)(j / S) & 1u, abort_flag, a.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, a.tok_tile);
      for (int it = 0; it < n_it; ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&full[s], ph, abort_flag, a.status)) break;
        tc_fence_after();
        const uint64_t ad = sdesc_sw128(smem_u32(smA + (size_t)s * kATileBytes));
        const uint64_t bd = sdesc_sw128(smem_u32(smB + (size_t)s * btile));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tmem_d, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
      }
      mma_commit(tmem_full);
    }
  } else {
    // ---------------- epilogue: warps 2..9, two per TMEM lane quarter (warp w
    // reads lanes 32 (w % 4)..), splitting the token columns in two halves
    const int q = warp & 3;
    const int e = warp - 2;       // 0..7
    const int hf = e >> 2;        // which half of the token columns (EW == 8)
    const int TT = a.tok_tile;
    const int c_lo = hf ? a.tok_half : 0, c_hi = (hf || EW == 4) ? TT : a.tok_half;
    const int n = n_tile * 128 + 32 * q + lane;
    // every epilogue warp takes the same decision
    if (lane == 0) votes[e] = (mbar_wait(tmem_full, 0, abort_flag, a.status) && !*abort_flag) ? 1 : 0;
    named_bar<1>(kEpiThreads);
    bool go = true;
#pragma unroll
    for (int i = 0; i < kEpiWarps; ++i) go = go && votes[i];
    pdl_wait();
    if (go && a.tma_out) {
      // TMEM -> 128-byte-swizzled staging in the drained pipeline buffers -> TMA stores
      tc_fence_after();
      uint8_t* stg = smem;
      const uint32_t trow = (uint32_t)(32 * q) << 16;
      if (a.e_mode == kEPartial) {
        // lane quarter q owns one box: [TT tokens][32 fp32] of output features 32q..32q+31
        uint8_t* box = stg + (size_t)q * TT * 128;
        const uint32_t lo = (uint32_t)((lane & 3) << 2);
        for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
          float v[16];
          tmem_ld16(tmem_d + trow + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c0 + j;
            *reinterpret_cast<float*>(box + t * 128 + ((((lane >> 2) ^ (t & 7))) << 4) + lo) = v[j];
          }
        }
        fence_proxy_async_smem();
        if (EW == 8) quarter_bar(q);  // both halves of the box are staged
        if (hf == 0 && lane == 0) {
          tma_store_3d(&omap, box, n_tile * 128 + 32 * q, t0, ks);
          bulk_commit();
          bulk_wait_read_all();
        }
        __syncwarp();
      } else if (a.e_mode == kEQkvRope) {
        // two boxes [TT tokens][64 bf16]: first and second members of the tile's 64 pairs
        const int half = a.dh >> 1;
        const int n0 = n_tile * 128;
        const int hb = n0 / a.dh;
        const int pair0 = (n0 - hb * a.dh) >> 1;
        const int p = n - hb * a.dh;
        const int pair = p >> 1, odd = p & 1;
        const int pl = pair - pair0;
        const bool rot = hb < a.n_rot_heads;
        uint8_t* box = stg + (size_t)odd * TT * 128;
        const uint32_t lo = (uint32_t)((pl & 7) << 1);
        float2 csn[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = t0 + c_lo + j;
          csn[j] = (rot && t < a.M) ? __ldg(a.rope_cs + (size_t)t * half + pair) : make_float2(1.f, 0.f);
        }
        for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
          float2 csv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) csv[j] = csn[j];
          if (c0 + 16 < c_hi) {  // table values of the next 16 tokens, loaded one step ahead
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = t0 + c0 + 16 + j;
              csn[j] = (rot && t < a.M) ? __ldg(a.rope_cs + (size_t)t * half + pair) : make_float2(1.f, 0.f);
            }
          }
          float v[16];
          tmem_ld16(tmem_d + trow + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            const int t = c0 + j;
            float outv = v[j];
            if (rot) {
              const float x1 = odd ? other : v[j], x2 = odd ? v[j] : other;
              outv = odd ? (x2 * csv[j].x + x1 * csv[j].y) : (x1 * csv[j].x - x2 * csv[j].y);
            }
            *reinterpret_cast<bf16*>(box + t * 128 + (((pl >> 3) ^ (t & 7)) << 4) + lo) =
                __float2bfloat16_rn(outv);
          }
        }
        fence_proxy_async_smem();
        named_bar<1>(kEpiThreads);
        if (threadIdx.x == 64) {
          tma_store_2d(&omap, stg, hb * a.dh + pair0, t0);
          tma_store_2d(&omap, stg + (size_t)TT * 128, hb * a.dh + half + pair0, t0);
          bulk_commit();
          bulk_wait_read_all();
        }
        __syncwarp();
      } else {  // kEGeglu: one box [TT tokens][64 bf16] of GeGLU outputs n/2
        // lane 2i holds gate j = 16q + i and lane 2i + 1 its up value; lane 4k
        // packs outputs 2k and 2k + 1 (from lane 4k + 2) into one 4-byte store
        const int jl = 16 * q + (lane >> 1);
        const uint32_t lo = (uint32_t)((jl & 7) << 1);
        for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
          float v[16];
          tmem_ld16(tmem_d + trow + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            const float r = gelu_tanh(v[j]) * other;  // meaningful on even lanes
            const float r_next = __shfl_down_sync(0xffffffffu, r, 2);
            const int t = c0 + j;
            if ((lane & 3) == 0)
              *reinterpret_cast<__nv_bfloat162*>(stg + t * 128 + (((jl >> 3) ^ (t & 7)) << 4) + lo) =
                  __floats2bfloat162_rn(r, r_next);
          }
        }
        fence_proxy_async_smem();
        named_bar<1>(kEpiThreads);
        if (threadIdx.x == 64) {
          tma_store_2d(&omap, stg, n_tile * 64, t0);
          bulk_commit();
          bulk_wait_read_all();
        }
        __syncwarp();
      }
    } else if (go) {
      tc_fence_after();
      for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
        float v[16];
        tmem_ld16(tmem_d + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
        if (a.e_mode == kEPartial) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = t0 + c0 + j;
            if (t < a.M) a.part[((size_t)ks * a.M + t) * a.N + n] = v[j];
          }
        } else if (a.e_mode == kEQkvRope) {
          const int half = a.dh >> 1;
          const int hb = n / a.dh, p = n - hb * a.dh;
          const int pair = p >> 1, odd = p & 1;
          const bool rot = hb < a.n_rot_heads;
          float2 csv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = t0 + c0 + j;
            csv[j] = (rot && t < a.M) ? __ldg(a.rope_cs + (size_t)t * half + pair) : make_float2(1.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            const int t = t0 + c0 + j;
            if (t < a.M) {
              float outv = v[j];
              if (rot) {
                const float2 cs = csv[j];
                const float x1 = odd ? other : v[j], x2 = odd ? v[j] : other;
                outv = odd ? (x2 * cs.x + x1 * cs.y) : (x1 * cs.x - x2 * cs.y);
              }
              a.out_bf16[(size_t)t * a.N + hb * a.dh + pair + odd * half] = __float2bfloat16_rn(outv);
            }
          }
        } else {  // kEGeglu
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            const int t = t0 + c0 + j;
            if (t < a.M && !(n & 1))
              a.out_bf16[(size_t)t * (a.N >> 1) + (n >> 1)] = __float2bfloat16_rn(gelu_tanh(v[j]) * other);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // the last commit tracks every MMA this CTA issued: wait for it before freeing TMEM
    if (*abort_flag && lane == 0) mbar_wait(tmem_full, 0, abort_flag, a.status);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_d, tmem_cols);
  }
}

// ---------------------------------------------------------------- between the GEMMs
// Sum the split-K partials of the merged QKV projection in split order, apply
// RoPE to q and k, store q|k|v in natural head layout.  One thread per rotation pair.
__global__ void k_reduce_qkv(const float* __restrict__ part, int ks_n, int M, int N, int dh,
                             int n_rot_heads, const float2* __restrict__ cs, bf16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const int np = N >> 1;
  if (idx >= (long)M * np) return;
  const int t = (int)(idx / np), pp = (int)(idx - (long)t * np);
  const int n = 2 * pp;
  float x1 = 0.f, x2 = 0.f;
  for (int j0 = 0; j0 < ks_n; j0 += 8) {  // eight splits in flight, summed in split order
    float2 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      v[j] = j0 + j < ks_n ? __ldcg(reinterpret_cast<const float2*>(part + ((size_t)(j0 + j) * M + t) * N + n))
                           : make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j0 + j < ks_n) {
        x1 += v[j].x;
        x2 += v[j].y;
      }
  }
  const int half = dh >> 1;
  const int hb = n / dh, pair = (n - hb * dh) >> 1;
  float o1 = x1, o2 = x2;
  if (hb < n_rot_heads) {
    const float2 c = cs[(size_t)t * half + pair];
    o1 = x1 * c.x - x2 * c.y;
    o2 = x2 * c.x + x1 * c.y;
  }
  out[(size_t)t * N + hb * dh + pair] = __float2bfloat16_rn(o1);
  out[(size_t)t * N + hb * dh + pair + half] = __float2bfloat16_rn(o2);
}

constexpr int kRowThreads = 256;

template <int NT>
__device__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += red[w];
  return t;
}

// One token row: h += gate * (sum of the split-K partials, in split order);
// then, if `scale` is given, y = adaRMS(h) with the next sublayer's
// (scale, shift) as the bf16 operand of the next GEMM.  A thread owns COLS
// columns and issues the loads of SB splits of all of them before it adds
// (a row costs about ceil(ks / SB) L2 round trips).
template <int NT, int COLS, int SB>
__global__ void __launch_bounds__(NT) k_resid_norm(const float* __restrict__ part, int ks_n, int M, int D,
                                                   float* __restrict__ h, const float* __restrict__ gate,
                                                   const float* __restrict__ scale,
                                                   const float* __restrict__ shift, float eps,
                                                   bf16* __restrict__ y) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[NT / 32];
  const int t = blockIdx.x;
  float* hr = h + (size_t)t * D;
  const size_t stride = (size_t)M * D;
  float ss = 0.f;
  for (int n0 = threadIdx.x; n0 < D; n0 += NT * COLS) {
    float acc[COLS];
    bool in[COLS];
#pragma unroll
    for (int e = 0; e < COLS; ++e) {
      acc[e] = 0.f;
      in[e] = n0 + e * NT < D;
    }
    const float* pp = part + (size_t)t * D + n0;
    for (int j0 = 0; j0 < ks_n; j0 += SB) {
      float v[SB][COLS];
#pragma unroll
      for (int j = 0; j < SB; ++j)
#pragma unroll
        for (int e = 0; e < COLS; ++e)
          v[j][e] = (j0 + j < ks_n && in[e]) ? __ldcg(pp + (size_t)(j0 + j) * stride + e * NT) : 0.f;
#pragma unroll
      for (int j = 0; j < SB; ++j)
#pragma unroll
        for (int e = 0; e < COLS; ++e)
          if (j0 + j < ks_n) acc[e] += v[j][e];
    }
#pragma unroll
    for (int e = 0; e < COLS; ++e) {
      if (!in[e]) continue;
      const int n = n0 + e * NT;
      const float hn = hr[n] + gate[n] * acc[e];
      hr[n] = hn;
      ss += hn * hn;
    }
  }
  if (scale == nullptr) return;
  ss = block_sum<NT>(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)D + eps);
  for (int n = threadIdx.x; n < D; n += NT)
    y[(size_t)t * D + n] = __float2bfloat16_rn(hr[n] * r * (1.f + scale[n]) + shift[n]);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float (&f)[8]) {
  const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(hv[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

// Action input projection h = x W_in^T + b_in of one token row, then the first
// layer's adaRMS into the bf16 operand of its QKV GEMM.  With A % 8 == 0 a
// thread reads its four W_in rows as 16-byte vectors, four of each at a time.
__global__ void __launch_bounds__(kRowThreads) k_inproj_norm(const float* __restrict__ x,
                                                            const bf16* __restrict__ w_in,
                                                            const bf16* __restrict__ b_in, int D, int A,
                                                            float* __restrict__ h,
                                                            const float* __restrict__ scale,
                                                            const float* __restrict__ shift, float eps,
                                                            bf16* __restrict__ y) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kRowThreads / 32];
  extern __shared__ float xs[];
  const int t = blockIdx.x;
  for (int k = threadIdx.x; k < A; k += kRowThreads) xs[k] = x[(size_t)t * A + k];
  __syncthreads();
  float* hr = h + (size_t)t * D;
  const int A8 = A / 8;
  const bool vec = (A & 7) == 0;
  float ss = 0.f;
  for (int n0 = threadIdx.x; n0 < D; n0 += 4 * kRowThreads) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (vec) {
      for (int kb = 0; kb < A8; kb += 4) {
        uint4 q[4][4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int n = n0 + e * kRowThreads;
            q[e][j] = (n < D && kb + j < A8) ? __ldg(reinterpret_cast<const uint4*>(w_in + (size_t)n * A) + kb + j)
                                             : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (kb + j >= A8) continue;
            float f[8];
            bf16x8_to_f32(q[e][j], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[e] += xs[8 * (kb + j) + i] * f[i];
          }
      }
    } else {
      for (int e = 0; e < 4; ++e) {
        const int n = n0 + e * kRowThreads;
        if (n < D)
          for (int k = 0; k < A; ++k) acc[e] += xs[k] * __bfloat162float(w_in[(size_t)n * A + k]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = n0 + e * kRowThreads;
      if (n >= D) continue;
      const float hn = acc[e] + __bfloat162float(b_in[n]);
      hr[n] = hn;
      ss += hn * hn;
    }
  }
  ss = block_sum<kRowThreads>(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)D + eps);
  for (int n = threadIdx.x; n < D; n += kRowThreads)
    y[(size_t)t * D + n] = __float2bfloat16_rn(hr[n] * r * (1.f + scale[n]) + shift[n]);
}

// GeGLU of the split-K partials of the interleaved gate/up projection:
// m[t][j] = gelu_tanh(sum g) * (sum u), sums in split order.
__global__ void k_geglu_reduce(const float* __restrict__ part, int ks_n, int M, int F,
                               bf16* __restrict__ m) {
  pdl_trigger();
  pdl_wait();
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)M * F) return;
  const int t = (int)(idx / F), j = (int)(idx - (long)t * F);
  float g = 0.f, u = 0.f;
  for (int s0 = 0; s0 < ks_n; s0 += 8) {  // eight splits in flight, summed in split order
    float2 v[8];
#pragma unroll
    for (int j2 = 0; j2 < 8; ++j2)
      v[j2] = s0 + j2 < ks_n
                  ? __ldcg(reinterpret_cast<const float2*>(part + ((size_t)(s0 + j2) * M + t) * 2 * F + 2 * j))
                  : make_float2(0.f, 0.f);
#pragma unroll
    for (int j2 = 0; j2 < 8; ++j2)
      if (s0 + j2 < ks_n) {
        g += v[j2].x;
        u += v[j2].y;
      }
  }
  m[idx] = __float2bfloat16_rn(gelu_tanh(g) * u);
}

}  // namespace

size_t tc_gemm_smem_bytes(int stages, int tok_tile) {
  return 1024 + (size_t)stages * (kATileBytes + (size_t)tok_tile * 128) + (2 * stages + 1) * 8 + 64;
}

GemmPlan plan_gemm(int N, int K, int M, int sm_count, int min_split, int max_split) {
  GemmPlan p;
  p.N = N;
  p.K = K;
  p.n_tiles = N / 128;
  p.tok_tiles = (M + 255) / 256;
  if (p.tok_tiles < 1) p.tok_tiles = 1;
  int tt = (M + p.tok_tiles - 1) / p.tok_tiles;
  tt = ((tt + 15) / 16) * 16;
  if (tt < 16) tt = 16;
  p.tok_tile = tt;
  p.kb_total = K / 64;
  const int base = p.n_tiles * p.tok_tiles;
  int ks = sm_count / base;
  if (max_split > 0 && ks > max_split) ks = max_split;
  if (ks < min_split) ks = min_split;
  if (ks < 1) ks = 1;
  if (ks > p.kb_total) ks = p.kb_total;
  p.ksplit = ks;
  int cols = 32;
  while (cols < tt) cols <<= 1;
  p.tmem_cols = cols;
  // as many stages as a CTA has K blocks, within the shared-memory budget
  const int per_cta = (p.kb_total + ks - 1) / ks;
  int stages = per_cta < 8 ? per_cta : 8;
  if (stages < 2) stages = 2;
  while (stages > 2 && tc_gemm_smem_bytes(stages, tt) > 200 * 1024) --stages;
  // the epilogue stages its output tile (up to tt x 128 fp32) in the drained pipeline buffers
  while ((size_t)stages * (kATileBytes + (size_t)tt * 128) < (size_t)tt * 512 && stages < 8) ++stages;
  p.stages = stages;
  p.smem = tc_gemm_smem_bytes(stages, tt);
  p.grid = base * ks;
  return p;
}

// Every kernel of the bf16 path asks for the same (maximum) shared-memory
// carve-out, so consecutive kernels never make an SM re-partition L1/shared.
template <typename K>
cudaError_t max_carveout(K kern) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

cudaError_t gemm_kernel_setup() {
  cudaError_t e = cudaFuncSetAttribute(k_tc_gemm<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_tc_gemm<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  if (e == cudaSuccess) e = max_carveout(k_tc_gemm<4>);
  if (e == cudaSuccess) e = max_carveout(k_tc_gemm<8>);
  if (e == cudaSuccess) e = max_carveout(k_reduce_qkv);
  if (e == cudaSuccess) e = max_carveout(k_resid_norm<256, 4, 8>);
  if (e == cudaSuccess) e = max_carveout(k_inproj_norm);
  if (e == cudaSuccess) e = max_carveout(k_geglu_reduce);
  return e;
}

cudaError_t launch_tc_gemm(const CUtensorMap& wmap, const CUtensorMap& amap, const GemmPlan& p,
                           TcGemmArgs a, cudaStream_t s, bool pdl) {
  a.N = p.N;
  a.K = p.K;
  a.tok_tile = p.tok_tile;
  a.n_tiles = p.n_tiles;
  a.tok_tiles = p.tok_tiles;
  a.ksplit = p.ksplit;
  a.kb_total = p.kb_total;
  a.stages = p.stages;
  a.tmem_cols = p.tmem_cols;
  a.tok_half = ((p.tok_tile / 2 + 15) / 16) * 16;
  CUtensorMap omap;
  memset(&omap, 0, sizeof(omap));
  a.tma_out = 0;
  cudaError_t e = cudaSuccess;
  if (a.e_mode == kEPartial) {
    e = make_f32_3d_map(&omap, a.part, p.N, a.M, p.ksplit, p.tok_tile);
    a.tma_out = 1;
  } else if (a.e_mode == kEQkvRope && a.dh >= 128) {
    e = make_bf16_map(&omap, a.out_bf16, a.out_rows, p.N, p.tok_tile);
    a.tma_out = 1;
  } else if (a.e_mode == kEGeglu) {
    e = make_bf16_map(&omap, a.out_bf16, a.out_rows, p.N / 2, p.tok_tile);
    a.tma_out = 1;
  }
  if (e != cudaSuccess) return e;
  if (p.tok_tile > 64)
    return launch_k(k_tc_gemm<8>, dim3(p.grid), dim3(kThreadsFor(8)), p.smem, s, pdl, wmap, amap, omap, a);
  return launch_k(k_tc_gemm<4>, dim3(p.grid), dim3(kThreadsFor(4)), p.smem, s, pdl, wmap, amap, omap, a);
}

cudaError_t launch_reduce_qkv(const float* part, int ks, int M, int N, int dh, int n_rot_heads,
                              const float2* cs, bf16* out, cudaStream_t s, bool pdl) {
  const long n = (long)M * (N / 2);
  return launch_k(k_reduce_qkv, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, pdl, part, ks, M,
                  N, dh, n_rot_heads, cs, out);
}

cudaError_t launch_resid_norm(const float* part, int ks, int M, int D, float* h, const float* gate,
                              const float* scale, const float* shift, float eps, bf16* y,
                              cudaStream_t s, bool pdl) {
  // 256 threads x 4 columns a row (measured faster than 1024 x 1 at 50 rows too)
  return launch_k(k_resid_norm<256, 4, 8>, dim3(M), dim3(256), 0, s, pdl, part, ks, M, D, h, gate, scale, shift,
                  eps, y);
}

cudaError_t launch_inproj_norm(const float* x, const bf16* w_in, const bf16* b_in, int M, int D,
                               int A, float* h, const float* scale, const float* shift, float eps,
                               bf16* y, cudaStream_t s, bool pdl) {
  return launch_k(k_inproj_norm, dim3(M), dim3(kRowThreads), A * sizeof(float), s, pdl, x, w_in,
                  b_in, D, A, h, scale, shift, eps, y);
}

cudaError_t launch_geglu_reduce(const float* part, int ks, int M, int F, bf16* m, cudaStream_t s,
                                bool pdl) {
  const long n = (long)M * F;
  return launch_k(k_geglu_reduce, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, pdl, part, ks,
                  M, F, m);
}

}  // namespace ae
