// Host side of the tcgen05 GEMMs (planner, launcher, the bf16-weight
// instantiations of k_tc_gemm) and the row kernels around them: the action
// input projection, the prefill's embedding norm and the adaRMS shift fold.
#include "ae_gemm_kernel.cuh"

namespace ae {
namespace {

using namespace tc;


__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float (&f)[8]) {
  const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(hv[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

constexpr int kRowThreads = 256;

// Action input projection h = x W_in^T + b_in of one token row (MolmoBot PR,
// Part 2; LoongForge Pi0.5 blog, section 5.3), then the first QKV GEMM's
// operand bf16(h * (1 + scale)) and the row's sums of h^2 per 128 features.
// With A % 8 == 0 a thread reads its four W_in rows as 16-byte vectors.
__global__ void __launch_bounds__(kRowThreads) k_inproj_norm(const float* __restrict__ x,
                                                            const bf16* __restrict__ w_in,
                                                            const bf16* __restrict__ b_in, int M, int D,
                                                            int A, float* __restrict__ h,
                                                            const float* __restrict__ scale,
                                                            bf16* __restrict__ aout,
                                                            float* __restrict__ ss_out) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float xs[];  // [A] then the row of h [D]
  float* hs = xs + A;
  const int t = blockIdx.x;
  for (int k = threadIdx.x; k < A; k += kRowThreads) xs[k] = x[(size_t)t * A + k];
  __syncthreads();
  float* hr = h + (size_t)t * D;
  const int A8 = A / 8;
  const bool vec = (A & 7) == 0;
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
      hs[n] = hn;
      aout[(size_t)t * D + n] = __float2bfloat16_rn(hn * (1.f + scale[n]));
    }
  }
  __syncthreads();
  // sums of squares per 128-feature tile, one warp per tile, fixed order
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int tile = warp; tile < D / 128; tile += kRowThreads / 32) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v = hs[tile * 128 + 32 * j + lane];
      ss += v * v;
    }
    ss = warp_sum(ss);
    if (lane == 0) ss_out[(size_t)tile * M + t] = ss;
  }
}

// Prefill input: h = emb of one token row, then the first QKV GEMM's operand
// bf16(h * (1 + scale)) and the row's sums of h^2 per 128 features.
__global__ void __launch_bounds__(kRowThreads) k_embed_norm(const bf16* __restrict__ emb, int M, int D,
                                                           float* __restrict__ h, const float* __restrict__ scale,
                                                           bf16* __restrict__ aout, float* __restrict__ ss_out) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float hs[];  // the row of h [D]
  const int t = blockIdx.x;
  for (int n = threadIdx.x; n < D; n += kRowThreads) {
    const float hn = __bfloat162float(emb[(size_t)t * D + n]);
    h[(size_t)t * D + n] = hn;
    hs[n] = hn;
    aout[(size_t)t * D + n] = __float2bfloat16_rn(hn * (1.f + scale[n]));
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int tile = warp; tile < D / 128; tile += kRowThreads / 32) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v = hs[tile * 128 + 32 * j + lane];
      ss += v * v;
    }
    ss = warp_sum(ss);
    if (lane == 0) ss_out[(size_t)tile * M + t] = ss;
  }
}

// fold[s][l][off + n] = sum_k W[l][n][k] * shift[s][l][k]: the constant that
// adaRMS's shift adds to every output feature n of a GEMM, for each flow step
// s and layer l (shift of norm `j` of the modulation table).  One warp per
// weight row; the row stays in registers across the steps.
__global__ void __launch_bounds__(256) k_fold_shift(const bf16* __restrict__ W, int N, int D,
                                                    const float* __restrict__ mod, int S, int L, int j,
                                                    float* __restrict__ fold, int nf, int off) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp, l = blockIdx.y;
  if (n >= N) return;
  const bf16* wr = W + ((size_t)l * N + n) * D;
  for (int s = 0; s < S; ++s) {
    const float* sh = mod + (((size_t)s * L + l) * 2 + j) * 3 * D + D;
    float acc = 0.f;
    for (int k0 = 8 * lane; k0 < D; k0 += 256) {
      float f[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(wr + k0), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc += f[i] * sh[k0 + i];
    }
    acc = warp_sum(acc);
    if (lane == 0) fold[((size_t)s * L + l) * nf + off + n] = acc;
  }
}

}  // namespace

size_t tc_gemm_smem_bytes(int stages, int tok_tile) {
  return 1024 + (size_t)stages * (kATileBytes + (size_t)tok_tile * 128) + (2 * stages + 1) * 8 + 64;
}

// Token tiling and pipeline depth shared by both planners.
static void plan_tiles(GemmPlan& p, int N, int K, int M, int tok_tiles = 0) {
  // a pipeline stage spans 64 K columns, 128 with e4m3 weights (p.wf set by the caller)
  p.N = N;
  p.K = K;
  p.n_tiles = N / 128;
  p.tok_tiles = tok_tiles > 0 ? tok_tiles : (M + 255) / 256;
  if (p.tok_tiles < 1) p.tok_tiles = 1;
  int tt = (M + p.tok_tiles - 1) / p.tok_tiles;
  tt = ((tt + 15) / 16) * 16;
  if (tt < 16) tt = 16;
  p.tok_tile = tt;
  p.kb_total = K / (64 * stage_width(p.wf));
  p.xbulk = 0;
  int cols = 32;
  while (cols < tt) cols <<= 1;
  p.tmem_cols = cols;
}

namespace {
// Clusters of `ks` CTAs of this configuration the GPU holds at once (cached
// per device and configuration).
int max_active_clusters(int ew, int ks, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, ew, ks, smem);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ks * 64));
  cfg.blockDim = dim3((unsigned)kThreadsFor(ew));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)ks;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = ew == 8 ? cudaOccupancyMaxActiveClusters(&n, k_tc_gemm<8, kEResid, 2, 0>, &cfg)
                                : cudaOccupancyMaxActiveClusters(&n, k_tc_gemm<4, kEResid, 2, 0>, &cfg);
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}
}  // namespace

GemmPlan plan_gemm_cl(int N, int K, int M, int sm_count, int max_split, bool retile, int exact_split, int wf) {
  GemmPlan p;
  p.wf = wf;
  // a fixed split keeps the token tiles at 128 so that the split-K receive
  // buffer (the fp32 tile) fits beside the pipeline whatever M is
  plan_tiles(p, N, K, M, exact_split > 0 ? (M + 127) / 128 : 0);
  // An unsplit GEMM that leaves SMs idle spends them on more, shorter token
  // tiles (down to 64 tokens) instead.
  if (retile && sm_count / (p.n_tiles * p.tok_tiles) <= 1) {
    int best = p.tok_tiles;
    for (int t = p.tok_tiles + 1; p.n_tiles * t <= sm_count; ++t) {
      const int tt = (((M + t - 1) / t + 15) / 16) * 16;
      if (tt < 64) break;
      best = t;
    }
    if (best != p.tok_tiles) plan_tiles(p, N, K, M, best);
  }
  const int ew = p.tok_tile > 64 ? 8 : 4;
  const int base = p.n_tiles * p.tok_tiles;
  int ks = exact_split > 0 ? exact_split : sm_count / base;
  if (max_split > 0 && ks > max_split) ks = max_split;
  if (ks > kMaxCluster) ks = kMaxCluster;
  if (ks > p.kb_total) ks = p.kb_total;
  if (ks < 1) ks = 1;
  // a split costs nothing only while every cluster of the launch is resident at once
  for (;; --ks) {
    p.ksplit = ks;
    // as many stages as a CTA has K blocks, within the shared-memory budget
    const int per_cta = (p.kb_total + ks - 1) / ks;
    int stages = per_cta < 8 ? per_cta : 8;
    if (stages < 2) stages = 2;
    // e4m3 stages are twice as wide: a long token tile with a split-K receive
    // buffer may leave room for one only (serial, but keeps the split)
    const int min_stages = wf ? 1 : 2;
    while (stages > min_stages && 1024 + gemm_smem_layout(stages, p.tok_tile, ks, wf).total > 220 * 1024) --stages;
    // split K by bulk copies stages the fp32 partial tile (tt x 128) in the
    // drained pipeline buffers; where it cannot fit, per-thread remote stores
    const size_t stage_need = (size_t)p.tok_tile * 512;
    auto fits = [&](int st) {
      return (size_t)st * stage_width(wf) * (kATileBytes + (size_t)p.tok_tile * 128) >= stage_need &&
             1024 + gemm_smem_layout(st, p.tok_tile, ks, wf).total <= 232448;
    };
    p.xbulk = 0;
    if (ks > 1)
      for (int st = stages; st <= 8; ++st)
        if (fits(st)) {
          stages = st;
          p.xbulk = 1;
          break;
        }
    p.stages = stages;
    p.smem = 1024 + gemm_smem_layout(stages, p.tok_tile, ks, wf).total;
    p.grid = base * ks;
    if (ks == 1 || exact_split > 0) break;
    if (p.smem <= 232448 && max_active_clusters(ew, ks, p.smem) >= base) break;
  }
  // An unsplit GEMM with between one and two waves of tiles keeps two CTAs
  // per SM (half the shared memory each, at most 256 TMEM columns each), so
  // every tile is resident at once and one CTA's epilogue runs under the
  // other's mainloop.
  if (p.ksplit == 1 && base > sm_count && base <= 2 * sm_count && p.tmem_cols <= 256) {
    while (p.stages > 2 && 1024 + gemm_smem_layout(p.stages, p.tok_tile, 1, wf).total > 113 * 1024) --p.stages;
    p.smem = 1024 + gemm_smem_layout(p.stages, p.tok_tile, 1, wf).total;
  }
  return p;
}

// Every bf16-weight instantiation of k_tc_gemm, in the order of gemm_kernel(ew, mode, xp).
template <typename F>
void for_each_gemm(F&& f) {
  f(k_tc_gemm<4, kEQkvRope, 0, 0>); f(k_tc_gemm<4, kEQkvRope, 1, 0>); f(k_tc_gemm<4, kEQkvRope, 2, 0>);
  f(k_tc_gemm<4, kEGeglu, 0, 0>); f(k_tc_gemm<4, kEGeglu, 1, 0>); f(k_tc_gemm<4, kEGeglu, 2, 0>);
  f(k_tc_gemm<4, kEResid, 0, 0>); f(k_tc_gemm<4, kEResid, 1, 0>); f(k_tc_gemm<4, kEResid, 2, 0>);
  f(k_tc_gemm<8, kEQkvRope, 0, 0>); f(k_tc_gemm<8, kEQkvRope, 1, 0>); f(k_tc_gemm<8, kEQkvRope, 2, 0>);
  f(k_tc_gemm<8, kEGeglu, 0, 0>); f(k_tc_gemm<8, kEGeglu, 1, 0>); f(k_tc_gemm<8, kEGeglu, 2, 0>);
  f(k_tc_gemm<8, kEResid, 0, 0>); f(k_tc_gemm<8, kEResid, 1, 0>); f(k_tc_gemm<8, kEResid, 2, 0>);
}

GemmKernel gemm_kernel(int ew, int mode, int xp) {
  GemmKernel table[18];
  int i = 0;
  for_each_gemm([&](auto kern) { table[i++] = kern; });
  const int m = mode == kEQkvRope ? 0 : (mode == kEGeglu ? 1 : 2);
  return table[(ew == 8 ? 9 : 0) + 3 * m + xp];
}

cudaError_t gemm_kernel_setup() {
  cudaError_t e = cudaSuccess;
  auto attrs = [&](auto kern) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  };
  for_each_gemm([&](auto kern) { attrs(kern); });
  if (e == cudaSuccess) e = gemm_kernel_setup_fp8();
  // every kernel of the bf16 path asks for the same (maximum) shared-memory
  // carve-out, so consecutive kernels never make an SM re-partition L1/shared
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_inproj_norm, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
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
  a.xbulk = p.xbulk;
  const int ew = p.tok_tile > 64 ? 8 : 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid, (unsigned)(a.z_count > 1 ? a.z_count : 1));
  cfg.blockDim = dim3((unsigned)kThreadsFor(ew));
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (pdl) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.ksplit > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = (unsigned)p.ksplit;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  const int xp = p.ksplit == 1 ? 0 : (p.xbulk ? 1 : 2);
  return cudaLaunchKernelEx(&cfg, p.wf ? gemm_kernel_fp8(ew, a.e_mode, xp) : gemm_kernel(ew, a.e_mode, xp), wmap,
                            amap, a);
}

cudaError_t launch_inproj_norm(const float* x, const bf16* w_in, const bf16* b_in, int M, int D, int A,
                               float* h, const float* scale, bf16* aout, float* ss_out, cudaStream_t s,
                               bool pdl) {
  return launch_k(k_inproj_norm, dim3(M), dim3(kRowThreads), (size_t)(A + D) * sizeof(float), s, pdl, x,
                  w_in, b_in, M, D, A, h, scale, aout, ss_out);
}

cudaError_t launch_embed_norm(const bf16* emb, int M, int D, float* h, const float* scale, bf16* aout,
                              float* ss_out, cudaStream_t s, bool pdl) {
  return launch_k(k_embed_norm, dim3(M), dim3(kRowThreads), (size_t)D * sizeof(float), s, pdl, emb, M, D, h, scale,
                  aout, ss_out);
}

cudaError_t launch_fold_shift(const bf16* W, int N, int D, const float* mod, int S, int L, int j, float* fold,
                              int nf, int off, cudaStream_t s) {
  return launch_k(k_fold_shift, dim3((unsigned)((N + 7) / 8), (unsigned)L), dim3(256), 0, s, false, W, N, D,
                  mod, S, L, j, fold, nf, off);
}

}  // namespace ae
