// tcgen05 GEMMs of the bf16 path, with the rest of the layer fused into their
// epilogues.
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
// Split K without a reduce kernel: the K splits of one output tile are the
// CTAs of one thread-block cluster, and the tile's tokens are dealt to them in
// runs of 4-token groups.  Each CTA sends every other CTA its partial of that
// CTA's run through distributed shared memory (one bulk copy per run out of
// the drained pipeline buffers, or, where the fp32 tile does not fit there,
// per-thread remote stores); the owner sums the cluster's partials in rank
// order (so the result does not depend on timing) and runs the epilogue on
// its run:
//   kEQkvRope   adaRMS folded in (below), RoPE (rotate_half pairs) on q and k,
//               bf16 q|k|v store
//   kEGeglu     adaRMS folded in, gelu_tanh(g) * u of the interleaved gate/up
//               rows, bf16 store
//   kEResid     gated residual h += gate * acc (LoongForge Pi0.5 blog,
//               section 2), then the next GEMM's operand bf16(h * (1 + scale))
//               and the tile's share of sum(h^2) per token
// adaRMS folded into the consumer: with y = h r (1 + scale) + shift and r the
// per-token reciprocal RMS, y W^T = r * ((h * (1 + scale)) W^T) + shift W^T.
// The producer of h writes h * (1 + scale) and per-128-feature sums of h^2;
// the consumer's epilogue forms r from those sums, scales its accumulator by
// r and adds the per-feature constant shift W^T, which the time table holds
// for every (flow step, layer).  No kernel waits for a whole-row norm.
//
// fp8 weights (WF = 1; MolmoBot PR, Part 3 and the LoongForge Pi0.5 blog,
// section 7: per-tensor e4m3 weights, the GEMM result restored by the
// tensor's scale): a pipeline stage spans 128 K columns instead of 64.  TMA
// brings the stage's 128-row x 128-column block of e4m3 codes (16 KB, one
// 128-byte row per weight row, as many row transfers as a bf16 block of half
// the width) into a staging buffer; the epilogue warps, idle during the
// mainloop, widen it exactly to bf16 as two 128-byte-swizzled 64-column
// tiles, which the MMA reads like two bf16 stages; the epilogue multiplies
// each output row by its tensor's dequantization factor before anything else.
#pragma once

#include <cuda_fp8.h>
#include <math.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "ae_internal.h"
#include "ae_tc.cuh"

namespace ae {
namespace {

using namespace tc;

// Warp 0 issues TMA, warp 1 MMA, warps 2.. run the epilogue: EW = 4 (one per
// TMEM lane quarter) for token tiles up to 64, EW = 8 (two per quarter, each
// taking half of the token columns) for longer tiles.
constexpr int kThreadsFor(int ew) { return 64 + 32 * ew; }
constexpr int kATileBytes = 128 * 128;  // 128 weight rows x 64 bf16
constexpr int kMaxCluster = 16;

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

// Split-K: the tokens of a tile are dealt to the ranks of its cluster in runs
// of whole 4-token groups; rank r emits tokens [run_lo(r), run_lo(r + 1)),
// the last run clipped to the tile's valid tokens.
__host__ __device__ inline int run_lo(int r, int ng, int ks) { return 4 * (r * ng / ks); }
// Tokens of the longest run: a rank's receive buffer holds the partials of its
// run from each rank, token-major: recv[src][token][128 features].
__host__ __device__ inline int recv_slice(int n_tok, int ks) { return 4 * (((n_tok + 3) / 4 + ks - 1) / ks); }

__host__ __device__ inline uint32_t recv_bytes(int tt, int ks) {
  return ks > 1 ? (uint32_t)ks * (uint32_t)recv_slice(tt, ks) * 512u : 0u;
}

// Shared-memory layout of k_tc_gemm, byte offsets from the 1024-aligned base:
// pipeline stages (weights, token tiles; after the mainloop they stage the
// fp32 partial tile), the split-K receive buffer, mbarriers and flags, the
// per-token reciprocal RMS of the emitted tokens and the per-quarter sums of
// squares.
// With fp8 weights a stage holds two 64-column weight and token tiles, the
// e4m3 block stages in its own buffer (`raw`), and each stage has two more
// barriers (codes landed, codes widened).
struct GemmSmem {
  uint32_t a, b, raw, recv, bars, rn, red, total;
};

constexpr int kRawTileBytes = 128 * 128;  // 128 weight rows x 128 e4m3 codes

// 64-column sub-blocks per pipeline stage
__host__ __device__ constexpr int stage_width(int wf) { return wf ? 2 : 1; }

__host__ __device__ inline GemmSmem gemm_smem_layout(int stages, int tt, int ks, int wf = 0) {
  GemmSmem L;
  const uint32_t sw = (uint32_t)stage_width(wf);
  L.a = 0;
  L.b = (uint32_t)stages * sw * kATileBytes;
  L.raw = L.b + (uint32_t)stages * sw * (uint32_t)(tt * 128);
  L.recv = L.raw + (wf ? (uint32_t)stages * kRawTileBytes : 0u);
  L.bars = L.recv + recv_bytes(tt, ks);
  L.rn = L.bars + (uint32_t)((wf ? 4 : 2) * stages + 2) * 8u + 64u;  // + TMEM base, abort flag, votes[8]
  L.red = L.rn + (256u + 16u) * 4u;
  L.total = L.red + 4u * 256u * 4u;
  return L;
}

// What the epilogue needs, copied out of the kernel arguments into registers.
struct Epi {
  int mode, M, N, n_ss, norm_dim, dh, half, n_rot_heads, TT;
  float eps;
  const float* ss_in;
  const float* fold;
  bf16* out;
  const float2* rope_cs;
  float* h;
  const float* gate;
  const float* scale_next;
  bf16* a_out;
  uint64_t keep;   // L2 evict-last policy for the RoPE table and the residual stream
  float* red;      // shared [4][TT]
  const float* rn; // shared, per emitted token
};

// Per-token inputs of one 4-token group that the epilogue of MODE reads from
// global memory (RoPE (cos, sin) of the thread's pair, or the residual h);
// loaded two groups ahead of use.
template <int MODE>
__device__ __forceinline__ void pre4(const Epi& E, int n, int tok0, int cnt, float2 (&aux)[4]) {
  if (MODE == kEQkvRope) {
    const int hb = n / E.dh, pair = (n - hb * E.dh) >> 1;
    const bool rot = hb < E.n_rot_heads;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      aux[j] = (rot && j < cnt) ? ld_keep_f2(E.rope_cs + (size_t)(tok0 + j) * E.half + pair, E.keep) : make_float2(1.f, 0.f);
  } else if (MODE == kEResid) {
#pragma unroll
    for (int j = 0; j < 4; ++j) aux[j].x = j < cnt ? ld_keep_f32(E.h + (size_t)(tok0 + j) * E.N + n, E.keep) : 0.f;
  }
}

// Epilogue of up to 4 consecutive emitted tokens of feature row n (token
// tok0.., index i0.. among this CTA's emitted tokens), values v = sums over K,
// aux = pre4 of the group.  All lanes of the warp call it with the same i0,
// tok0 and cnt (shuffles inside).  Small on purpose: it runs in a rolled loop.
template <int MODE>
__device__ __forceinline__ void emit4(const Epi& E, int n, int q, int lane, int i0, int tok0, const float (&v)[4],
                                      int cnt, float cf, float gt, float sc, const float2 (&aux)[4]) {
  if (MODE == kEResid) {
    float hn[4], sq[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hn[j] = aux[j].x + gt * v[j];
      sq[j] = j < cnt ? hn[j] * hn[j] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < cnt) {
        E.h[(size_t)(tok0 + j) * E.N + n] = hn[j];
        if (E.scale_next != nullptr) E.a_out[(size_t)(tok0 + j) * E.N + n] = __float2bfloat16_rn(hn[j] * (1.f + sc));
      }
    // per-token sum over the warp by a transposed butterfly: lanes with bit 4
    // clear keep tokens 0, 1, then lanes with bit 3 clear keep the first of
    // the two; lane l ends with token 2 b4 + b3
    {
      const bool up = lane & 16;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float got = __shfl_xor_sync(0xffffffffu, up ? sq[k] : sq[2 + k], 16);
        sq[k] = (up ? sq[2 + k] : sq[k]) + got;
      }
    }
    const bool up8 = lane & 8;
    float s = (up8 ? sq[1] : sq[0]) + __shfl_xor_sync(0xffffffffu, up8 ? sq[0] : sq[1], 8);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    const int t = 2 * ((lane >> 4) & 1) + ((lane >> 3) & 1);
    if ((lane & 7) == 0 && t < cnt) E.red[q * E.TT + i0 + t] = s;
  } else if (MODE == kEGeglu) {
    // lane 2i holds gate row i, lane 2i + 1 its up row; the even lane takes
    // tokens 0, 1 of the group, the odd lane tokens 2, 3
    float x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = E.rn[i0 + j] * v[j] + cf;
    const bool odd = lane & 1;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float got = __shfl_xor_sync(0xffffffffu, odd ? x[k] : x[2 + k], 1);
      const float g = odd ? got : x[k], u = odd ? x[2 + k] : got;
      const int j = odd ? 2 + k : k;
      if (j < cnt) E.out[(size_t)(tok0 + j) * (E.N >> 1) + (n >> 1)] = __float2bfloat16_rn(gelu_tanh(g) * u);
    }
  } else {  // kEQkvRope: packed rows 2j, 2j + 1 of a head are its dims j, j + dh/2
    const int hb = n / E.dh, p = n - hb * E.dh;
    const int pair = p >> 1, odd = p & 1;
    const bool rot = hb < E.n_rot_heads;
    bf16* ocol = E.out + hb * E.dh + pair + odd * E.half;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x = E.rn[i0 + j] * v[j] + cf;
      const float other = __shfl_xor_sync(0xffffffffu, x, 1);
      float o = x;
      if (rot) o = odd ? (x * aux[j].x + other * aux[j].y) : (x * aux[j].x - other * aux[j].y);
      if (j < cnt) ocol[(size_t)(tok0 + j) * E.N] = __float2bfloat16_rn(o);
    }
  }
}

// pre4 for a 16-token chunk (more independent work per warp on long token
// runs), loaded one chunk ahead of use.
template <int MODE>
__device__ __forceinline__ void pre16(const Epi& E, int n, int tok0, int cnt, float2 (&aux)[16]) {
  if (MODE == kEQkvRope) {
    const int hb = n / E.dh, pair = (n - hb * E.dh) >> 1;
    const bool rot = hb < E.n_rot_heads;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      aux[j] = (rot && j < cnt) ? ld_keep_f2(E.rope_cs + (size_t)(tok0 + j) * E.half + pair, E.keep) : make_float2(1.f, 0.f);
  } else if (MODE == kEResid) {
#pragma unroll
    for (int j = 0; j < 16; ++j) aux[j].x = j < cnt ? ld_keep_f32(E.h + (size_t)(tok0 + j) * E.N + n, E.keep) : 0.f;
  }
}

// Epilogue of up to 16 consecutive emitted tokens of feature row n (token
// tok0.., index i0.. among this CTA's emitted tokens), values v = sums over K,
// aux = pre16 of the chunk.  All lanes of the warp call it with the same i0,
// tok0 and cnt (shuffles inside); every load precedes every store.
template <int MODE>
__device__ __forceinline__ void emit16(const Epi& E, int n, int q, int lane, int i0, int tok0,
                                       const float (&v)[16], int cnt, float cf, float gt, float sc,
                                       const float2 (&aux)[16]) {
  if (MODE == kEResid) {
    float hn[16], sq[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      hn[j] = aux[j].x + gt * v[j];
      sq[j] = j < cnt ? hn[j] * hn[j] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < cnt) {
        E.h[(size_t)(tok0 + j) * E.N + n] = hn[j];
        if (E.scale_next != nullptr) E.a_out[(size_t)(tok0 + j) * E.N + n] = __float2bfloat16_rn(hn[j] * (1.f + sc));
      }
    // sum of sq over the warp for each of the 16 tokens by a transposed
    // butterfly: after the step with mask m, lanes with bit m clear keep the
    // lower half of their vector; lane l ends with token 8b4 + 4b3 + 2b2 + b1
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const bool up = lane & 16;
      const float send = up ? sq[k] : sq[8 + k];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      sq[k] = (up ? sq[8 + k] : sq[k]) + got;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const bool up = lane & 8;
      const float send = up ? sq[k] : sq[4 + k];
      const float got = __shfl_xor_sync(0xffffffffu, send, 8);
      sq[k] = (up ? sq[4 + k] : sq[k]) + got;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const bool up = lane & 4;
      const float send = up ? sq[k] : sq[2 + k];
      const float got = __shfl_xor_sync(0xffffffffu, send, 4);
      sq[k] = (up ? sq[2 + k] : sq[k]) + got;
    }
    {
      const bool up = lane & 2;
      const float send = up ? sq[0] : sq[1];
      const float got = __shfl_xor_sync(0xffffffffu, send, 2);
      sq[0] = (up ? sq[1] : sq[0]) + got;
    }
    const float tot = sq[0] + __shfl_xor_sync(0xffffffffu, sq[0], 1);
    const int t = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
    if (!(lane & 1) && t < cnt) E.red[q * E.TT + i0 + t] = tot;
  } else if (MODE == kEGeglu) {
    // lane 2i holds gate row i, lane 2i + 1 its up row, for 16 tokens; the
    // pair splits the tokens: the even lane takes tokens 0..7, the odd one 8..15
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = E.rn[i0 + j];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = x[j] * v[j] + cf;
    const bool odd = lane & 1;
    float r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float got = __shfl_xor_sync(0xffffffffu, odd ? x[k] : x[8 + k], 1);
      const float g = odd ? got : x[k], u = odd ? x[8 + k] : got;
      r[k] = gelu_tanh(g) * u;
    }
    bf16* ocol = E.out + (n >> 1);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int j = odd ? 8 + k : k;
      if (j < cnt) ocol[(size_t)(tok0 + j) * (E.N >> 1)] = __float2bfloat16_rn(r[k]);
    }
  } else {  // kEQkvRope: packed rows 2j, 2j + 1 of a head are its dims j, j + dh/2
    const int hb = n / E.dh, p = n - hb * E.dh;
    const int pair = p >> 1, odd = p & 1;
    const bool rot = hb < E.n_rot_heads;
    float x[16], o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = E.rn[i0 + j];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = x[j] * v[j] + cf;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, x[j], 1);
      o[j] = x[j];
      if (rot) o[j] = odd ? (x[j] * aux[j].x + other * aux[j].y) : (x[j] * aux[j].x - other * aux[j].y);
    }
    bf16* ocol = E.out + hb * E.dh + pair + odd * E.half;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < cnt) ocol[(size_t)(tok0 + j) * E.N] = __float2bfloat16_rn(o[j]);
  }
}

template <int N>
__device__ __forceinline__ void scale_rows(float (&v)[N], float ws) {
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] *= ws;
}

// Two e4m3 codes (low byte first) as a bf16 pair: e4m3 -> f16 is exact (every
// e4m3 value is a normal f16), f16 -> f32 is exact, and f32 -> bf16 keeps the
// value (at most 4 significant bits, exponents -9..8).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(__half2(h));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Widen one weight row of a staged e4m3 block (128 codes in a 128-byte row,
// 16-byte chunk ci at ci ^ (row % 8): TMA's 128-byte swizzle) into its rows of
// the two bf16 operand tiles of the stage (64 columns, 128 bytes a row each,
// same swizzle, the layout the MMA's descriptors name).  The 16 codes of input
// chunk ci become chunks 2 (ci % 4) and 2 (ci % 4) + 1 of tile ci / 4.  Lanes
// hold consecutive rows, so each group of 8 lanes reads and writes 8
// different bank quads.
__device__ __forceinline__ void widen_e4m3_row(const uint8_t* src_row, uint8_t* dst_row0, int row) {
  const int rho = row & 7;
#pragma unroll
  for (int ci = 0; ci < 8; ++ci) {
    const uint4 in = *reinterpret_cast<const uint4*>(src_row + ((ci ^ rho) << 4));
    uint8_t* dst_row = dst_row0 + (ci >> 2) * kATileBytes;
    const int cc = ci & 3;
    uint4 o0, o1;
    o0.x = e4m3x2_to_bf16x2(in.x);
    o0.y = e4m3x2_to_bf16x2(in.x >> 16);
    o0.z = e4m3x2_to_bf16x2(in.y);
    o0.w = e4m3x2_to_bf16x2(in.y >> 16);
    o1.x = e4m3x2_to_bf16x2(in.z);
    o1.y = e4m3x2_to_bf16x2(in.z >> 16);
    o1.z = e4m3x2_to_bf16x2(in.w);
    o1.w = e4m3x2_to_bf16x2(in.w >> 16);
    *reinterpret_cast<uint4*>(dst_row + (((2 * cc) ^ rho) << 4)) = o0;
    *reinterpret_cast<uint4*>(dst_row + (((2 * cc + 1) ^ rho) << 4)) = o1;
  }
}

// One instantiation per epilogue MODE and split-K exchange XP (0 unsplit,
// 1 bulk copies, 2 per-thread remote stores): each launch carries only the
// code it runs, which at batch 1 runs once per CTA from a cold instruction cache.
template <int EW, int MODE, int XP, int WF>
__global__ void __launch_bounds__(kThreadsFor(EW), 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap amap,
              const __grid_constant__ TcGemmArgs a) {
  constexpr int kEpiWarps = EW;
  constexpr int kEpiThreads = 32 * EW;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = a.stages;
  const int TT = a.tok_tile;
  constexpr int SW = stage_width(WF);  // 64-column sub-blocks per stage
  const int btile = TT * 128;          // one 64-column token tile
  const int ksn = a.ksplit;
  const GemmSmem L = gemm_smem_layout(S, TT, ksn, WF);
  uint8_t* smA = smem + L.a;
  uint8_t* smB = smem + L.b;
  uint8_t* smW8 = smem + L.raw;  // fp8 weights: staged e4m3 blocks
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + S;
  uint64_t* tmem_full = empty + S;
  uint64_t* recv_bar = tmem_full + 1;  // split K: this rank's partials from every rank have landed
  // fp8 weights: full[s] then counts the token tile only; wfull[s] the e4m3
  // block, wide[s] its bf16 form (one arrival per widening warp)
  uint64_t* wfull = recv_bar + 1;
  uint64_t* wide = wfull + S;
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(WF ? wide + S : recv_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_p + 1);
  volatile int* votes = reinterpret_cast<volatile int*>(tmem_base_p + 2);  // [kEpiWarps]
  float* rn_s = reinterpret_cast<float*>(smem + L.rn);                      // [<= 256 + 16]
  float* red_s = reinterpret_cast<float*>(smem + L.red);                    // [4][TT]
  const float* recv = reinterpret_cast<const float*>(smem + L.recv);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the K splits of one output tile are consecutive CTAs forming one cluster
  const int ks = ksn > 1 ? (int)cluster_rank() : 0;
  const int idx = blockIdx.x / ksn;
  const int n_tile = idx % a.n_tiles;
  const int tt = idx / a.n_tiles;
  const int kb_begin = (int)((long)ks * a.kb_total / ksn);
  const int kb_end = (int)((long)(ks + 1) * a.kb_total / ksn);
  const int n_it = kb_end - kb_begin;
  const int t0 = tt * TT;
  const int nv = min(TT, a.M - t0);  // valid tokens of the tile
  // Tokens this CTA emits: the whole tile when unsplit, else its rank's run
  // of 4-token groups.
  const int ng = (nv + 3) >> 2;
  const int e_lo = run_lo(ks, ng, ksn);
  const int e_hi = min(run_lo(ks + 1, ng, ksn), nv);
  const int slice = recv_slice(nv, ksn);
  auto kcol = [&](int it) { return (kb_begin + it) * 64 * SW; };
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      if (WF) {
        mbar_init(&wfull[s], 1);
        mbar_init(&wide[s], 4);
      }
    }
    mbar_init(tmem_full, 1);
    mbar_init(recv_bar, 1);
    // bulk exchange: every rank sends this rank its partials of our run
    if (XP == 1) mbar_arrive_expect_tx(recv_bar, (uint32_t)(ksn * (e_hi - e_lo) * 512));
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
  // peers may write into this CTA once its receive barrier is initialised
  if constexpr (XP != 0) cluster_arrive();
  const uint32_t tmem_d = *tmem_base_p;
  bool go = false;
  // epilogue role (warps 2..): TMEM lane quarter, column half, feature row
  const int q = warp & 3;
  const int hf = (warp - 2) >> 2;
  const int f = 32 * q + lane;
  const int n = n_tile * 128 + f;
  Epi E;
  E.mode = a.e_mode;
  E.M = a.M;
  E.N = a.N;
  E.n_ss = a.n_ss;
  E.norm_dim = a.norm_dim;
  E.dh = a.dh;
  E.half = a.dh >> 1;
  E.n_rot_heads = a.n_rot_heads;
  E.TT = TT;
  E.eps = a.eps;
  E.ss_in = a.ss_in;
  E.fold = a.fold;
  // gridDim.y > 1: independent GEMMs of the same shape, z-th one offset in the
  // stacked weight, the stacked operand and the output (layers of a stack)
  const int z = blockIdx.y;
  E.out = a.out_bf16 + (size_t)z * a.z_out;
  E.rope_cs = a.rope_cs;
  E.h = a.h;
  E.gate = a.gate;
  E.scale_next = a.scale_next;
  E.a_out = a.a_out;
  E.red = red_s;
  E.rn = rn_s;
  E.keep = policy_evict_last();
  float* const ss_out = a.ss_out;
  int* const status = a.status;
  float cf = 0.f, gt = 0.f, sc = 0.f;
  float ws = 1.f;  // fp8 weights: dequantization factor of feature row n's tensor
  float2 aux0[4], aux1[4];  // per-token inputs of the next two 4-token groups (epilogue warps)
  // token columns this warp reads from TMEM (unsplit: also the ones it emits)
  const int c_lo = hf ? a.tok_half : 0;
  const int c_hi = min((hf || EW == 4) ? TT : a.tok_half, nv);
  // split K: tokens of this rank's run that this warp emits after the reduction
  const int ns = e_hi - e_lo;
  const int p_mid = EW == 8 ? 4 * ((ns + 7) / 8) : ns;
  const int p_lo = hf ? p_mid : 0, p_hi = hf ? ns : p_mid;
  const uint32_t trow = (uint32_t)(32 * q) << 16;

  if (warp == 0) {
    // ---------------- TMA producer: weight slab + token tile per 64-wide K block
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&amap);
      // a weight slab read by one token tile is not read again this flow step:
      // evict it first; with several token tiles the other tiles' CTAs read it
      // moments later, so it keeps the normal policy
      const uint64_t pol_w = a.tok_tiles > 1 ? policy_evict_normal() : policy_evict_first();
      const int row = a.w_row0 + z * a.z_w_rows + n_tile * 128;
      // the token box may hold only the valid rows of a single short tile
      const uint32_t bytes = (WF ? 0u : (uint32_t)kATileBytes) + SW * (uint32_t)(a.act_rows > 0 ? a.act_rows : TT) * 128u;
      // Weights do not depend on the previous kernel: fill the first stages and
      // start pulling this slab of the next layer into L2 before waiting on it.
      const int pre = n_it < S ? n_it : S;
      for (int it = 0; it < pre; ++it) {
        if (WF) {
          mbar_arrive_expect_tx(&wfull[it], kRawTileBytes);
          tma_load_2d(smW8 + (size_t)it * kRawTileBytes, &wmap, &wfull[it], kcol(it), row, pol_w);
        } else {
          mbar_arrive_expect_tx(&full[it], bytes);
          tma_load_2d(smA + (size_t)it * kATileBytes, &wmap, &full[it], kcol(it), row, pol_w);
        }
      }
      if (a.w_next_row0 >= 0)
        for (int it = 0; it < n_it; ++it)
          tma_prefetch_l2_2d(&wmap, kcol(it), a.w_next_row0 + n_tile * 128);
      pdl_wait();
      for (int it = 0; it < pre; ++it) {
        if (WF) mbar_arrive_expect_tx(&full[it], bytes);
#pragma unroll
        for (int j = 0; j < SW; ++j)
          tma_load_2d_nohint(smB + ((size_t)it * SW + j) * btile, &amap, &full[it], kcol(it) + 64 * j,
                             a.act_row0 + z * a.z_act_rows + t0);
      }
      int it = pre;
      for (; it < n_it; ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, a.status)) break;
        const int kc = kcol(it);
        if (WF) {
          mbar_arrive_expect_tx(&wfull[s], kRawTileBytes);
          tma_load_2d(smW8 + (size_t)s * kRawTileBytes, &wmap, &wfull[s], kc, row, pol_w);
          mbar_arrive_expect_tx(&full[s], bytes);
        } else {
          mbar_arrive_expect_tx(&full[s], bytes);
          tma_load_2d(smA + (size_t)s * kATileBytes, &wmap, &full[s], kc, row, pol_w);
        }
#pragma unroll
        for (int j = 0; j < SW; ++j)
          tma_load_2d_nohint(smB + ((size_t)s * SW + j) * btile, &amap, &full[s], kc + 64 * j,
                             a.act_row0 + z * a.z_act_rows + t0);
      }
      // drain: no copy may still be in flight when the CTA exits (stages
      // already consumed pass at once; the wait holds even after an abort)
      for (int j = it - S > 0 ? it - S : 0; j < it; ++j) {
        mbar_drain(&full[j % S], (uint32_t)(j / S) & 1u, a.status);
        if (WF) mbar_drain(&wfull[j % S], (uint32_t)(j / S) & 1u, a.status);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, TT);
      for (int it = 0; it < n_it; ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait(&full[s], ph, abort_flag, a.status)) break;
        if (WF && !mbar_wait(&wide[s], ph, abort_flag, a.status)) break;
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < SW; ++j) {
          const uint64_t ad = sdesc_sw128(smem_u32(smA + ((size_t)s * SW + j) * kATileBytes));
          const uint64_t bd = sdesc_sw128(smem_u32(smB + ((size_t)s * SW + j) * btile));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(tmem_d, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(tmem_full);
    }
  } else {
    // ---------------- epilogue warps 2..: warp w reads TMEM lanes 32 (w % 4)..
    // (feature rows f); with EW == 8 the two warps of a lane quarter take the
    // two halves of the token columns.
    const int e = warp - 2;
    const int et = threadIdx.x - 64;
    // per-feature constants come from the time table (ready before this kernel)
    if constexpr (MODE == kEResid) {
      gt = E.gate[n];
      if (E.scale_next != nullptr) sc = E.scale_next[n];
    } else {
      cf = E.fold != nullptr ? E.fold[n] : 0.f;
    }
    if constexpr (WF != 0) {
      ws = a.w_scale[a.w_row0 + z * a.z_w_rows + n];
      // widen the staged e4m3 blocks as they land (the first ones were
      // requested before the producer waited on the previous kernel), one
      // weight row a lane; every lane's wait must succeed before any widens.
      // Pipeline stage s belongs to the four warps of group s % (EW / 4)
      // for every pass over the ring: a parity wait is only sound while the
      // waiter has seen the barrier's previous phase complete, which the
      // group's own program order guarantees (with an odd stage count,
      // groups taking alternate iterations would wait on a phase two ahead)
      const int row = et & 127;
      const int grp = e >> 2;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % S;
        if (s % (EW / 4) != grp) continue;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        const bool ok = mbar_wait(&wfull[s], ph, abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) break;
        widen_e4m3_row(smW8 + (size_t)s * kRawTileBytes + row * 128, smA + (size_t)s * SW * kATileBytes + row * 128,
                       row);
        fence_proxy_async_smem();  // the MMA reads the tiles through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&wide[s]);
      }
    }
    pdl_wait();
    // reciprocal RMS of the emitted tokens, while the mainloop runs
    if constexpr (MODE != kEResid)
      for (int i = et; i < e_hi - e_lo; i += kEpiThreads) {
        const int tok = t0 + e_lo + i;
        float ss = 0.f;
        for (int j = 0; j < E.n_ss; ++j) ss += E.ss_in[(size_t)j * E.M + tok];
        rn_s[i] = E.n_ss > 0 ? 1.0f / sqrtf(ss / (float)E.norm_dim + E.eps) : 1.f;  // n_ss 0: no norm
      }
    // the first two groups' per-token inputs, issued before the accumulator is ready
    {
      const int lo = XP == 0 ? c_lo : e_lo + p_lo, hi = XP == 0 ? c_hi : e_lo + p_hi;
      if constexpr (MODE == kEQkvRope) {
        if (lo < hi) pre4<kEQkvRope>(E, n, t0 + lo, min(4, hi - lo), aux0);
        if (lo + 4 < hi) pre4<kEQkvRope>(E, n, t0 + lo + 4, min(4, hi - lo - 4), aux1);
      } else if constexpr (MODE == kEResid) {
        if (lo < hi) pre4<kEResid>(E, n, t0 + lo, min(4, hi - lo), aux0);
        if (lo + 4 < hi) pre4<kEResid>(E, n, t0 + lo + 4, min(4, hi - lo - 4), aux1);
      }
    }
    if (lane == 0) votes[e] = (mbar_wait(tmem_full, 0, abort_flag, status) && !*abort_flag) ? 1 : 0;
    named_bar<1>(kEpiThreads);
    go = true;
#pragma unroll
    for (int i = 0; i < kEpiWarps; ++i) go = go && votes[i];
    if (go) {
      tc_fence_after();
      if constexpr (XP == 0) {
        // unsplit: the accumulator is the sum; emit straight from TMEM, 4 tokens a step
        auto run = [&]() {
          if constexpr (MODE == kEQkvRope) {
            // Long tiles of a rotated head: the tile's slice of the RoPE table
            // (tokens x its 64 pairs, 512 bytes a token) is copied once into
            // the drained pipeline buffers, every thread's 16-byte pieces in
            // flight together, instead of one round trip per 16-token chunk.
            const int hb0 = (n_tile * 128) / E.dh;
            const bool stage = E.dh >= 128 && hb0 < E.n_rot_heads && nv >= 64 &&
                               (size_t)TT * 512 <= (size_t)S * SW * (kATileBytes + (size_t)btile);
            if (stage) {
              float2* cs_s = reinterpret_cast<float2*>(smem);
              const int pair0 = (n_tile * 128 - hb0 * E.dh) >> 1;
              for (int i = threadIdx.x - 64; i < nv * 32; i += kEpiThreads) {
                const int t = i >> 5, c = i & 31;
                cp_async16(cs_s + t * 64 + 2 * c, E.rope_cs + (size_t)(t0 + t) * E.half + pair0 + 2 * c, 16);
              }
              cp_async_commit();
              cp_async_wait<0>();
              named_bar<1>(kEpiThreads);
              const int pl = ((n - hb0 * E.dh) >> 1) - pair0;  // this thread's pair within the slice
#pragma unroll 1
              for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
                float2 cur[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) cur[j] = cs_s[(c0 + j) * 64 + pl];
                float v[16];
                tmem_ld16(tmem_d + trow + (uint32_t)c0, v);
                if constexpr (WF != 0) scale_rows(v, ws);
                emit16<MODE>(E, n, q, lane, c0, t0 + c0, v, min(16, c_hi - c0), cf, gt, sc, cur);
              }
              return;
            }
          }
          if (c_hi - c_lo >= 32) {
            // long run: 16 tokens a step, next chunk's inputs one step ahead
            float2 nx[16];
            pre16<MODE>(E, n, t0 + c_lo, min(16, c_hi - c_lo), nx);
#pragma unroll 1
            for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
              float2 cur[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) cur[j] = nx[j];
              if (c0 + 16 < c_hi) pre16<MODE>(E, n, t0 + c0 + 16, min(16, c_hi - c0 - 16), nx);
              float v[16];
              tmem_ld16(tmem_d + trow + (uint32_t)c0, v);
              if constexpr (WF != 0) scale_rows(v, ws);
              emit16<MODE>(E, n, q, lane, c0, t0 + c0, v, min(16, c_hi - c0), cf, gt, sc, cur);
            }
            return;
          }
#pragma unroll 1
          for (int c0 = c_lo; c0 < c_hi; c0 += 4) {
            float2 cur[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              cur[j] = aux0[j];
              aux0[j] = aux1[j];
            }
            if (c0 + 8 < c_hi) pre4<MODE>(E, n, t0 + c0 + 8, min(4, c_hi - c0 - 8), aux1);
            float v[4];
            tmem_ld4(tmem_d + trow + (uint32_t)c0, v);
            if constexpr (WF != 0) scale_rows(v, ws);
            emit4<MODE>(E, n, q, lane, c0, t0 + c0, v, min(4, c_hi - c0), cf, gt, sc, cur);
          }
        };
        run();
      } else if constexpr (XP == 1) {
        // split K: stage this partial token-major in the drained pipeline
        // buffers, then send each rank its run of tokens with one bulk copy
        float* stg = reinterpret_cast<float*>(smem);
        if constexpr (EW == 4) {
          // a tile of at most 64 tokens: every column in one TMEM load and one wait
          float v[64];
          tmem_ld64(tmem_d + trow, v);
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (j < c_hi) stg[j * 128 + f] = v[j];
        } else {
#pragma unroll 1
          for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
            float v[16];
            tmem_ld16(tmem_d + trow + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) stg[(c0 + j) * 128 + f] = v[j];
          }
        }
        fence_proxy_async_smem();
      }
    }
    if constexpr (XP != 0) {
      cluster_wait();  // every rank of the cluster has started and initialised its barrier
      if constexpr (XP == 1) {
        named_bar<1>(kEpiThreads);
        // one lane per destination rank issues that rank's copy
        if (go && warp == 2) {
          const uint32_t stg_u = smem_u32(smem);
          const uint32_t dst0 = smem_u32(smem + L.recv) + (uint32_t)(ks * slice) * 512u;
          const uint32_t bar_u = smem_u32(recv_bar);
          for (int r = lane; r < ksn; r += 32) {
            const int lo = run_lo(r, ng, ksn), hi = min(run_lo(r + 1, ng, ksn), nv);
            if (hi <= lo) continue;
            bulk_to_peer(mapa(dst0, (uint32_t)r), stg_u + (uint32_t)lo * 512u, (uint32_t)(hi - lo) * 512u,
                         mapa(bar_u, (uint32_t)r));
          }
          bulk_commit();
        }
      } else {
        // the fp32 tile does not fit the pipeline buffers: each thread stores
        // its partials straight into the owners' receive buffers, 128
        // contiguous bytes per token and warp
        if (go) {
          const uint32_t recv_u = smem_u32(smem + L.recv) + (uint32_t)(ks * slice * 128 + f) * 4u;
#pragma unroll 1
          for (int c0 = c_lo; c0 < c_hi; c0 += 4) {
            float v[4];
            tmem_ld4(tmem_d + trow + (uint32_t)c0, v);
            const int r = ((c0 / 4 + 1) * ksn - 1) / ng;  // run_lo(r) <= c0 < run_lo(r + 1)
            const uint32_t a0 = mapa(recv_u + (uint32_t)(c0 - run_lo(r, ng, ksn)) * 512u, (uint32_t)r);
#pragma unroll
            for (int k = 0; k < 4; ++k) st_cluster_f32(a0 + 512u * k, v[k]);
          }
        }
        cluster_arrive();  // this rank's partials are written
      }
    }
  }
  if (warp < 2) {
    __syncwarp();
    if constexpr (XP != 0) {
      cluster_wait();
      if constexpr (XP == 2) {
        cluster_arrive();
        cluster_wait();
      }
    }
  }
  if constexpr (XP != 0) {
    if (XP == 2 && warp >= 2) cluster_wait();  // every rank's partials have been written
    if (XP == 1 && warp >= 2 && go) {
      // this rank's run from every rank (bounded wait)
      int ok = 1;
      if (lane == 0) ok = mbar_wait(recv_bar, 0, abort_flag, status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      go = ok != 0;
    }
    if (warp >= 2 && go) {
      // sum this rank's tokens over the cluster's partials in rank order, emit them
      auto run = [&]() {
        if (MODE != kEResid && p_hi - p_lo >= 16) {
          // long run: 16 tokens a step, four ranks' loads in flight
          float2 nx[16];
          pre16<MODE>(E, n, t0 + e_lo + p_lo, min(16, p_hi - p_lo), nx);
#pragma unroll 1
          for (int c0 = p_lo; c0 < p_hi; c0 += 16) {
            float2 cur[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) cur[j] = nx[j];
            if (c0 + 16 < p_hi) pre16<MODE>(E, n, t0 + e_lo + c0 + 16, min(16, p_hi - c0 - 16), nx);
            const int cnt = min(16, p_hi - c0);
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
            const float* rp = recv + (size_t)c0 * 128 + f;
            const size_t sstride = (size_t)slice * 128;
#pragma unroll 1
            for (int src = 0; src < ksn; src += 2) {
              float x[2][16];
#pragma unroll
              for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int j = 0; j < 16; ++j) x[u][j] = (src + u < ksn && j < cnt) ? rp[(src + u) * sstride + j * 128] : 0.f;
#pragma unroll
              for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += x[u][j];
            }
            if constexpr (WF != 0) scale_rows(v, ws);
            emit16<MODE>(E, n, q, lane, c0, t0 + e_lo + c0, v, cnt, cf, gt, sc, cur);
          }
          return;
        }
#pragma unroll 1
        for (int c0 = p_lo; c0 < p_hi; c0 += 4) {
          float2 cur[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            cur[j] = aux0[j];
            aux0[j] = aux1[j];
          }
          if (c0 + 8 < p_hi) pre4<MODE>(E, n, t0 + e_lo + c0 + 8, min(4, p_hi - c0 - 8), aux1);
          const int cnt = min(4, p_hi - c0);
          float v[4] = {0.f, 0.f, 0.f, 0.f};
          const float* rp = recv + (size_t)c0 * 128 + f;
          const size_t sstride = (size_t)slice * 128;
          int src = 0;
          for (; src + 4 <= ksn; src += 4) {  // four ranks' loads in flight, added in rank order
            float x[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int j = 0; j < 4; ++j) x[u][j] = j < cnt ? rp[(src + u) * sstride + j * 128] : 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int j = 0; j < 4; ++j) v[j] += x[u][j];
          }
          for (; src < ksn; ++src)
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] += j < cnt ? rp[src * sstride + j * 128] : 0.f;
          if constexpr (WF != 0) scale_rows(v, ws);
          emit4<MODE>(E, n, q, lane, c0, t0 + e_lo + c0, v, cnt, cf, gt, sc, cur);
        }
      };
      run();
    }
  }
  if (MODE == kEResid && warp >= 2) {
    // per-token sum of h^2 over the tile's 128 features (four lane quarters, in order)
    named_bar<2>(kEpiThreads);
    if (go && ss_out != nullptr)
      for (int i = threadIdx.x - 64; i < e_hi - e_lo; i += kEpiThreads)
        ss_out[(size_t)n_tile * E.M + t0 + e_lo + i] =
            (red_s[i] + red_s[TT + i]) + (red_s[2 * TT + i] + red_s[3 * TT + i]);
  }
  // the bulk copies out of the staging must have read it before the CTA exits
  if (XP == 1 && warp == 2) bulk_wait_read_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // the last commit tracks every MMA this CTA issued: wait for it before freeing TMEM
    if (*abort_flag && lane == 0) mbar_drain(tmem_full, 0, a.status);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_d, tmem_cols);
  }
}

}  // namespace
}  // namespace ae
