// tcgen05 GEMMs of the bf16 path with the layer's elementwise work fused in.
//
// Swap-AB: a CTA computes a 128-row slab of a weight matrix against a tile of
// up to 256 action tokens, D[n, t] = sum_k W[n, k] X[t, k].  The weight rows
// are the MMA's M = 128 operand (streamed by TMA into 128-byte-swizzled shared
// memory, evict-first in L2: each weight is read once per flow step), the
// token tile is the MMA's N operand, so a 50-token chunk costs a 64-wide
// tile instead of a 128-row one.  The accumulator lives in TMEM.
//
// The token operand is produced by threads, so the layer's prologue is fused:
//   kBRms    adaRMS of the fp32 residual stream (LoongForge Pi0.5 blog,
//            section 2: rms over the row, (1 + scale), + shift), cast to bf16;
//   kBCopy   a bf16 activation (attention output, GeGLU output);
//   kBGeglu  GeGLU of split-K partials of the merged gate/up projection.
// The epilogue fuses what follows the projection:
//   kEQkvRope   RoPE (rotate_half pairs) on q and k, bf16 store of q|k|v;
//   kEResid     gated residual h += gate * acc and the adaRMS sum of squares;
//   kEGeglu     gelu_tanh(g) * u from the merged gate/up rows;
//   kEPartial   fp32 split-K partials, summed in a fixed order later.
// Merged Q/K/V and gate/up weights follow sglang PR #34599, item 1.
#include <math.h>

#include "ae_internal.h"
#include "ae_tc.cuh"

namespace ae {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kProducerThreads = 192;  // warps 2..7
constexpr int kATileBytes = 128 * 128; // 128 weight rows x 64 bf16

__device__ __forceinline__ float gelu_tanh(float g) {
  return 0.5f * g * (1.f + tanhf(0.7978845608028654f * (g + 0.044715f * g * g * g)));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Produce the 8 bf16 values of token tg, features k..k+7 of the token operand.
__device__ __forceinline__ uint4 produce_chunk(const TcGemmArgs& a, int tg, int k, float r) {
  uint4 out;
  if (a.b_mode == kBCopy) {
    out = *reinterpret_cast<const uint4*>(a.act + (size_t)tg * a.K + k);
  } else if (a.b_mode == kBRms) {
    const float4* hp = reinterpret_cast<const float4*>(a.h + (size_t)tg * a.K + k);
    const float4* sp = reinterpret_cast<const float4*>(a.scale + k);
    const float4* tp = reinterpret_cast<const float4*>(a.shift + k);
    float x[8], s[8], t[8];
    *reinterpret_cast<float4*>(x) = hp[0];
    *reinterpret_cast<float4*>(x + 4) = hp[1];
    *reinterpret_cast<float4*>(s) = sp[0];
    *reinterpret_cast<float4*>(s + 4) = sp[1];
    *reinterpret_cast<float4*>(t) = tp[0];
    *reinterpret_cast<float4*>(t + 4) = tp[1];
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = x[e] * r * (1.f + s[e]) + t[e];
    out = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                     pack_bf16(y[6], y[7]));
  } else {  // kBGeglu: partial rows hold (g_j, u_j) pairs
    float g[8], u[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = u[e] = 0.f;
    for (int j = 0; j < a.gu_ks; ++j) {
      const float4* p =
          reinterpret_cast<const float4*>(a.gu_part + ((size_t)j * a.M + tg) * a.gu_ld + 2 * k);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = p[q];
        g[2 * q] += v.x;
        u[2 * q] += v.y;
        g[2 * q + 1] += v.z;
        u[2 * q + 1] += v.w;
      }
    }
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = gelu_tanh(g[e]) * u[e];
    out = make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                     pack_bf16(y[6], y[7]));
  }
  return out;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ TcGemmArgs a) {
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
  float* rms = reinterpret_cast<float*>(tmem_base_p + 4);       // [tok_tile]
  float* red = rms + a.tok_tile;                                  // [4][16] + 4 votes

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

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1 + kProducerThreads / 32);
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
    // ---------------- weight producer (TMA)
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      const uint64_t pol = policy_evict_first();
      const int row = a.w_row0 + n_tile * 128;
      int it = 0;
      for (; it < n_it; ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, a.status)) break;
        mbar_arrive_expect_tx(&full[s], kATileBytes);
        tma_load_2d(smA + (size_t)s * kATileBytes, &wmap, &full[s], (kb_begin + it) * 64, row, pol);
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
    // ---------------- token-operand producers (warps 2..7)
    const int ptid = threadIdx.x - 64;
    if (a.b_mode == kBRms) {
      for (int t = ptid; t < a.tok_tile; t += kProducerThreads) {
        const int tg = t0 + t;
        float r = 0.f;
        if (tg < a.M) {
          float ss = 0.f;
          for (int j = 0; j < a.n_sumsq; ++j) ss += a.sumsq[(size_t)j * a.M + tg];
          r = 1.0f / sqrtf(ss / (float)a.K + a.eps);
        }
        rms[t] = r;
      }
      named_bar(1, kProducerThreads);
    }
    for (int it = 0; it < n_it; ++it) {
      const int s = it % S;
      const uint32_t ph = (uint32_t)(it / S) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1u, abort_flag, a.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint8_t* bs = smB + (size_t)s * btile;
      const int kb = kb_begin + it;
      for (int c = ptid; c < a.tok_tile * 8; c += kProducerThreads) {
        const int t = c >> 3, ch = c & 7;
        const int tg = t0 + t;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tg < a.M) v = produce_chunk(a, tg, kb * 64 + ch * 8, rms[t]);
        *reinterpret_cast<uint4*>(bs + sw128_offset(t, ch)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
    }

    // ---------------- epilogue (warps 4..7: TMEM lanes 32*(warp%4) ..)
    if (warp >= 4) {
      const int q = warp & 3;
      const int rowl = 32 * q + lane;
      const int n = n_tile * 128 + rowl;
      // every epilogue warp takes the same decision: a mismatch would leave a
      // named barrier below waiting forever
      volatile int* votes = reinterpret_cast<volatile int*>(red + 64);
      if (lane == 0) votes[q] = (mbar_wait(tmem_full, 0, abort_flag, a.status) && !*abort_flag) ? 1 : 0;
      named_bar(3, 128);
      const bool go = votes[0] && votes[1] && votes[2] && votes[3];
      if (go) {
        tc_fence_after();
        for (int c0 = 0; c0 < a.tok_tile; c0 += 16) {
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
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
              const int t = t0 + c0 + j;
              if (t < a.M) {
                float outv = v[j];
                if (rot) {
                  const float2 cs = a.rope_cs[(size_t)t * half + pair];
                  const float x1 = odd ? other : v[j], x2 = odd ? v[j] : other;
                  outv = odd ? (x2 * cs.x + x1 * cs.y) : (x1 * cs.x - x2 * cs.y);
                }
                a.out_bf16[(size_t)t * a.N + hb * a.dh + pair + odd * half] = __float2bfloat16_rn(outv);
              }
            }
          } else if (a.e_mode == kEGeglu) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
              const int t = t0 + c0 + j;
              if (t < a.M && !(n & 1))
                a.out_bf16[(size_t)t * (a.N >> 1) + (n >> 1)] = __float2bfloat16_rn(gelu_tanh(v[j]) * other);
            }
          } else {  // kEResid
            const float g = a.gate[n];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = t0 + c0 + j;
              float sq = 0.f;
              if (t < a.M) {
                float* hp = a.h_out + (size_t)t * a.N + n;
                const float hn = *hp + g * v[j];
                *hp = hn;
                sq = hn * hn;
              }
              sq = warp_sum(sq);
              if (lane == 0) red[q * 16 + j] = sq;
            }
            named_bar(2, 128);
            if (q == 0 && lane < 16) {
              const int t = t0 + c0 + lane;
              if (t < a.M)
                a.sumsq_out[(size_t)n_tile * a.M + t] =
                    red[lane] + red[16 + lane] + red[32 + lane] + red[48 + lane];
            }
            named_bar(2, 128);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // the last commit tracks every MMA this CTA issued: wait for it before freeing TMEM
    if (*abort_flag) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(tmem_full, 0, abort_flag, a.status);
      __syncwarp();
      (void)ok;
    }
    tc_fence_after();
    tmem_dealloc(tmem_d, tmem_cols);
  }
}

// ---------------------------------------------------------------- split-K reductions
// Sum the split-K partials of the merged QKV projection in split order, apply
// RoPE to q and k, store q|k|v in natural head layout.  One thread per rotation pair.
__global__ void k_reduce_qkv(const float* __restrict__ part, int ks_n, int M, int N, int dh,
                             int n_rot_heads, const float2* __restrict__ cs, bf16* __restrict__ out) {
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const int np = N >> 1;
  if (idx >= (long)M * np) return;
  const int t = (int)(idx / np), pp = (int)(idx - (long)t * np);
  const int n = 2 * pp;
  float x1 = 0.f, x2 = 0.f;
  for (int j = 0; j < ks_n; ++j) {
    const float2 v = *reinterpret_cast<const float2*>(part + ((size_t)j * M + t) * N + n);
    x1 += v.x;
    x2 += v.y;
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

// Sum split-K partials in split order, gated residual, adaRMS sum of squares
// per 128-feature tile.  Block = one (feature tile, token).
__global__ void __launch_bounds__(128) k_reduce_resid(const float* __restrict__ part, int ks_n,
                                                      int M, int N, float* __restrict__ h,
                                                      const float* __restrict__ gate,
                                                      float* __restrict__ sumsq) {
  const int tile = blockIdx.x, t = blockIdx.y;
  const int n = tile * 128 + threadIdx.x;
  float s = 0.f;
  for (int j = 0; j < ks_n; ++j) s += part[((size_t)j * M + t) * N + n];
  float* hp = h + (size_t)t * N + n;
  const float hn = *hp + gate[n] * s;
  *hp = hn;
  __shared__ float wsum[4];
  float sq = warp_sum(hn * hn);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = sq;
  __syncthreads();
  if (threadIdx.x == 0) sumsq[(size_t)tile * M + t] = wsum[0] + wsum[1] + wsum[2] + wsum[3];
}

// Action input projection h = x W_in^T + b_in, plus the sum of squares per
// 128-feature tile for the first adaRMS.  Block = one (feature tile, token).
__global__ void __launch_bounds__(128) k_inproj_tc(const float* __restrict__ x,
                                                   const bf16* __restrict__ w_in,
                                                   const bf16* __restrict__ b_in, float* __restrict__ h,
                                                   float* __restrict__ sumsq, int M, int D, int A) {
  const int tile = blockIdx.x, t = blockIdx.y;
  const int n = tile * 128 + threadIdx.x;
  float s = 0.f;
  for (int k = 0; k < A; ++k) s += x[(size_t)t * A + k] * __bfloat162float(w_in[(size_t)n * A + k]);
  const float hn = s + __bfloat162float(b_in[n]);
  h[(size_t)t * D + n] = hn;
  __shared__ float wsum[4];
  float sq = warp_sum(hn * hn);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = sq;
  __syncthreads();
  if (threadIdx.x == 0) sumsq[(size_t)tile * M + t] = wsum[0] + wsum[1] + wsum[2] + wsum[3];
}

}  // namespace

size_t tc_gemm_smem_bytes(int stages, int tok_tile) {
  return 1024 + (size_t)stages * (kATileBytes + (size_t)tok_tile * 128) + (2 * stages + 1) * 8 +
         16 + (size_t)tok_tile * 4 + 68 * 4;
}

GemmPlan plan_gemm(int N, int K, int M, int sm_count, bool allow_split) {
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
  int ks = allow_split ? sm_count / base : 1;
  if (ks < 1) ks = 1;
  if (ks > p.kb_total) ks = p.kb_total;
  p.ksplit = ks;
  int cols = 32;
  while (cols < tt) cols <<= 1;
  p.tmem_cols = cols;
  int stages = 8;
  while (stages > 2 && tc_gemm_smem_bytes(stages, tt) > 220 * 1024) --stages;
  p.stages = stages;
  p.smem = tc_gemm_smem_bytes(stages, tt);
  p.grid = base * ks;
  return p;
}

cudaError_t launch_tc_gemm(const CUtensorMap& map, const GemmPlan& p, TcGemmArgs a, cudaStream_t s) {
  a.N = p.N;
  a.K = p.K;
  a.tok_tile = p.tok_tile;
  a.n_tiles = p.n_tiles;
  a.tok_tiles = p.tok_tiles;
  a.ksplit = p.ksplit;
  a.kb_total = p.kb_total;
  a.stages = p.stages;
  a.tmem_cols = p.tmem_cols;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_tc_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         232448);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k_tc_gemm<<<p.grid, kThreads, p.smem, s>>>(map, a);
  return cudaGetLastError();
}

void launch_reduce_qkv(const float* part, int ks, int M, int N, int dh, int n_rot_heads,
                       const float2* cs, bf16* out, cudaStream_t s) {
  const long n = (long)M * (N / 2);
  k_reduce_qkv<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(part, ks, M, N, dh, n_rot_heads, cs, out);
}

void launch_reduce_resid(const float* part, int ks, int M, int N, float* h, const float* gate,
                         float* sumsq, cudaStream_t s) {
  k_reduce_resid<<<dim3(N / 128, M), 128, 0, s>>>(part, ks, M, N, h, gate, sumsq);
}

void launch_inproj_tc(const float* x, const bf16* w_in, const bf16* b_in, float* h, float* sumsq,
                      int M, int D, int A, cudaStream_t s) {
  k_inproj_tc<<<dim3(D / 128, M), 128, 0, s>>>(x, w_in, b_in, h, sumsq, M, D, A);
}

}  // namespace ae
