// e4m3 weights of the block Linears (MolmoBot PR, Part 3: per-tensor fp8 on
// the fused QKV, attention output, gate/up and down Linears, amax -> scale ->
// cast, the GEMM result restored by the scale; LoongForge Pi0.5 blog, section
// 7: TorchAO's tensorwise recipe).  Here: the quantizer ae_create runs once
// over the packed weights, the adaRMS shift fold over codes, and the
// instantiations of k_tc_gemm that stream codes and widen them to bf16 in
// shared memory.
//
// Per tensor: amax = max |w|; s = fp32(448 / amax) (1 when amax = 0); code =
// e4m3(fp32(w * s)), rounded to nearest even and saturated at 448; the factor
// r = fp32(1 / s) multiplies the tensor's GEMM outputs.  Every step is one
// IEEE fp32 operation, so the codes depend on the weights alone.
#include "ae_gemm_kernel.cuh"

namespace ae {
namespace {

using namespace tc;

constexpr int kTensorsPerLayer = 7;  // wq, wk, wv, wo, wg, wu, wd

// Tensor (0..6) of row r of one layer of a packed matrix.
__device__ __forceinline__ int row_tensor(const RowGroups& g, int r) {
  if (g.kind == 1) return g.t0 + (r & 1);
  return g.t0 + (r >= g.b1 ? 1 : 0) + (r >= g.b2 ? 1 : 0);
}

// One warp per weight row: the row's max |w| into its tensor's slot.  The
// magnitudes are non-negative, so their bit patterns order like their values
// and an unsigned atomicMax on the bits is a float max.
__global__ void __launch_bounds__(256) k_tensor_amax(const bf16* __restrict__ W, int L, int K, RowGroups g,
                                                     float* __restrict__ amax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long row = (long)blockIdx.x * 8 + warp;
  if (row >= (long)L * g.rows) return;
  const int l = (int)(row / g.rows), r = (int)(row % g.rows);
  const bf16* w = W + row * K;
  float m = 0.f;
  for (int k0 = 8 * lane; k0 < K; k0 += 256) {
    const uint4 q = *reinterpret_cast<const uint4*>(w + k0);
    const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = __bfloat1622float2(hv[i]);
      m = fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0)
    atomicMax(reinterpret_cast<unsigned int*>(amax) + l * kTensorsPerLayer + row_tensor(g, r), __float_as_uint(m));
}

__global__ void k_tensor_scales(const float* __restrict__ amax, int n, float* __restrict__ s_out,
                                float* __restrict__ r_out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = amax[i];
  const float sc = a > 0.f ? __fdiv_rn(448.f, a) : 1.f;
  s_out[i] = sc;
  r_out[i] = __fdiv_rn(1.f, sc);
}

// One block per weight row: codes of the row, and the row's factor r.
__global__ void __launch_bounds__(128) k_quantize_e4m3(const bf16* __restrict__ W, int K, RowGroups g,
                                                       const float* __restrict__ s_slot,
                                                       const float* __restrict__ r_slot, uint8_t* __restrict__ codes,
                                                       float* __restrict__ row_r) {
  const long row = blockIdx.x;
  const int l = (int)(row / g.rows), r = (int)(row % g.rows);
  const int slot = l * kTensorsPerLayer + row_tensor(g, r);
  const float sc = s_slot[slot];
  if (threadIdx.x == 0) row_r[row] = r_slot[slot];
  const bf16* w = W + row * K;
  uint8_t* out = codes + row * K;
  for (int k0 = 8 * threadIdx.x; k0 < K; k0 += 8 * 128) {
    const uint4 q = *reinterpret_cast<const uint4*>(w + k0);
    const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&q);
    uint32_t packed[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 v = __bfloat1622float2(hv[i]);
      const float2 x = make_float2(__fmul_rn(v.x, sc), __fmul_rn(v.y, sc));
      const uint32_t two = (uint32_t)__nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
      if (i & 1) packed[i >> 1] |= two << 16;
      else packed[i >> 1] = two;
    }
    *reinterpret_cast<uint2*>(out + k0) = make_uint2(packed[0], packed[1]);
  }
}

// k_fold_shift over e4m3 codes: fold[s][l][off + n] = r[n] * sum_k
// e4m3(W8[l][n][k]) * shift[s][l][k], one warp per weight row.
__global__ void __launch_bounds__(256) k_fold_shift_e4m3(const uint8_t* __restrict__ W8,
                                                         const float* __restrict__ row_r, int N, int D,
                                                         const float* __restrict__ mod, int S, int L, int j,
                                                         float* __restrict__ fold, int nf, int off) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp, l = blockIdx.y;
  if (n >= N) return;
  const uint8_t* wr = W8 + ((size_t)l * N + n) * D;
  const float rr = row_r[(size_t)l * N + n];
  for (int s = 0; s < S; ++s) {
    const float* sh = mod + (((size_t)s * L + l) * 2 + j) * 3 * D + D;
    float acc = 0.f;
    for (int k0 = 8 * lane; k0 < D; k0 += 256) {
      const uint2 q = *reinterpret_cast<const uint2*>(wr + k0);
      const uint32_t wd[2] = {q.x, q.y};
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t two = (wd[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
        const float2 v = __half22float2(__half2(h));
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
      }
      // the bf16 fold's order: with weights that are codes times a power of
      // two, both folds give the same bits up to that power
#pragma unroll
      for (int i = 0; i < 8; ++i) acc += f[i] * sh[k0 + i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) fold[((size_t)s * L + l) * nf + off + n] = rr * acc;
  }
}

// Every e4m3-weight instantiation of k_tc_gemm, in the order of gemm_kernel_fp8(ew, mode, xp).
template <typename F>
void for_each_gemm_fp8(F&& f) {
  f(k_tc_gemm<4, kEQkvRope, 0, 1>); f(k_tc_gemm<4, kEQkvRope, 1, 1>); f(k_tc_gemm<4, kEQkvRope, 2, 1>);
  f(k_tc_gemm<4, kEGeglu, 0, 1>); f(k_tc_gemm<4, kEGeglu, 1, 1>); f(k_tc_gemm<4, kEGeglu, 2, 1>);
  f(k_tc_gemm<4, kEResid, 0, 1>); f(k_tc_gemm<4, kEResid, 1, 1>); f(k_tc_gemm<4, kEResid, 2, 1>);
  f(k_tc_gemm<8, kEQkvRope, 0, 1>); f(k_tc_gemm<8, kEQkvRope, 1, 1>); f(k_tc_gemm<8, kEQkvRope, 2, 1>);
  f(k_tc_gemm<8, kEGeglu, 0, 1>); f(k_tc_gemm<8, kEGeglu, 1, 1>); f(k_tc_gemm<8, kEGeglu, 2, 1>);
  f(k_tc_gemm<8, kEResid, 0, 1>); f(k_tc_gemm<8, kEResid, 1, 1>); f(k_tc_gemm<8, kEResid, 2, 1>);
}

}  // namespace

GemmKernel gemm_kernel_fp8(int ew, int mode, int xp) {
  GemmKernel table[18];
  int i = 0;
  for_each_gemm_fp8([&](auto kern) { table[i++] = kern; });
  const int m = mode == kEQkvRope ? 0 : (mode == kEGeglu ? 1 : 2);
  return table[(ew == 8 ? 9 : 0) + 3 * m + xp];
}

cudaError_t gemm_kernel_setup_fp8() {
  cudaError_t e = cudaSuccess;
  for_each_gemm_fp8([&](auto kern) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  return e;
}

cudaError_t launch_tensor_amax(const bf16* W, int L, int K, RowGroups g, float* amax, cudaStream_t s) {
  const long rows = (long)L * g.rows;
  return launch_k(k_tensor_amax, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, s, false, W, L, K, g, amax);
}

cudaError_t launch_tensor_scales(const float* amax, int n, float* s_out, float* r_out, cudaStream_t st) {
  return launch_k(k_tensor_scales, dim3((unsigned)((n + 127) / 128)), dim3(128), 0, st, false, amax, n, s_out, r_out);
}

cudaError_t launch_quantize_e4m3(const bf16* W, int L, int K, RowGroups g, const float* s_slot, const float* r_slot,
                                 uint8_t* codes, float* row_r, cudaStream_t st) {
  return launch_k(k_quantize_e4m3, dim3((unsigned)((long)L * g.rows)), dim3(128), 0, st, false, W, K, g, s_slot,
                  r_slot, codes, row_r);
}

cudaError_t launch_fold_shift_e4m3(const uint8_t* W8, const float* row_r, int N, int D, const float* mod, int S,
                                   int L, int j, float* fold, int nf, int off, cudaStream_t s) {
  return launch_k(k_fold_shift_e4m3, dim3((unsigned)((N + 7) / 8), (unsigned)L), dim3(256), 0, s, false, W8, row_r,
                  N, D, mod, S, L, j, fold, nf, off);
}

}  // namespace ae
