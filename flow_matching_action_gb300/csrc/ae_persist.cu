// The bf16 denoise loop as ONE persistent kernel per ae_sample: one CTA per
// SM runs every phase of every layer of every flow step; phases are separated
// by a bounded software grid barrier instead of kernel boundaries.
//
// A flow step is the same sequence of phases as the per-kernel path (MolmoBot
// PR, Part 2: the prefix binding is reused, only the action rows and t move):
//   in-proj + adaRMS1 | per layer: QKV GEMM (+RoPE) [| QKV split-K sum + RoPE]
//   | attention | chunk combine | O GEMM | sum + gated residual + adaRMS2
//   | gate/up GEMM (+GeGLU) [| GeGLU of the partials] | down GEMM
//   | sum + gated residual + next adaRMS1 | ... | final adaRMS + out-proj + Euler.
// At batch 1 a kernel boundary costs more than most of these phases, so here
// TMEM is allocated once, and each GEMM's first weight tiles are issued into
// the free pipeline buffers before the barrier that precedes it (weights do
// not depend on the previous phase), overlapping the weight stream with the
// barrier and the phase before.  Work units (GEMM tiles, attention chunk
// ranges, rows) are dealt to the CTAs round robin in a fixed order and every
// sum runs in a fixed order, so results do not depend on timing.
#include <math.h>
#include <string.h>

#include "ae_internal.h"
#include "ae_tc.cuh"

namespace ae {
namespace {

using namespace tc;

constexpr int kPT = 256;        // threads per CTA
constexpr int kMaxStages = 8;   // GEMM pipeline stages: P.stages (<= 8) for every GEMM of a launch
constexpr int kATile = 128 * 128;
constexpr int kChunk = 64;      // attention keys per chunk
constexpr int kSkip = -0x40000000;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleMargin = 8.f;
constexpr int kCodeChunks = 16;  // attention chunks whose gather codes a CTA keeps for the launch

// Control block (after the data region and the row scratch).
struct Ctrl {
  uint64_t full[kMaxStages], empty[kMaxStages], tmem_full;
  uint64_t bar_s, bar_o, bar_q, bar_kv[2];
  uint32_t tmem_base;
  int abort;
  int flag;
  int pad;
  float red[kPT / 32];
  int idx[2][kChunk];
  // Gather codes of this CTA's attention chunks (the same every layer and
  // step), filled once per launch when they fit: codes[slot][key in chunk],
  // slot_row[slot] = first prefix row of a chunk of 64 contiguous prefix rows
  // (loaded by TMA) or -1 (gathered).
  int n_cached;  // chunks cached, or -1
  int slot_row[kCodeChunks];
  int codes[kCodeChunks][kChunk];
};

__device__ __forceinline__ float gelu_tanh(float g) {
  return 0.5f * g * (1.f + tanhf(0.7978845608028654f * (g + 0.044715f * g * g * g)));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Per-CTA running counters; each lives in the threads that use it, so every
// mbarrier keeps counting phases across units, phases, layers and steps.
struct State {
  unsigned gen;        // grid barriers passed (thread 0)
  uint32_t pit;        // GEMM k-blocks issued (thread 0)
  uint32_t mit;        // GEMM k-blocks consumed (thread 32)
  uint32_t units;      // GEMM units finished (epilogue threads)
  int pre_gi, pre_layer, prefetched;  // weight tiles issued ahead of a GEMM phase (thread 0)
  uint32_t q_uses, s_uses, kv_ph[2];  // attention barrier phases (attention threads)
  int kv_pend[2], q_pend;             // attention copies not yet waited for (attention thread 0)
  int kv_pre;                         // the first chunk of the next attention phase was issued early
};

struct Ctx {
  uint8_t* smem;   // 1024-aligned data region (pipeline stages / attention tiles / staging)
  float* rows;     // row scratch: max(D, A) floats
  Ctrl* ctrl;
  uint32_t tmem;   // TMEM base (512 columns)
};

__device__ __forceinline__ volatile int* abort_flag(const Ctx& c) { return &c.ctrl->abort; }

// All 32 lanes of a warp wait together for the phase of `parity` of `bar`.
// A role that only one lane could run (issuing TMA or MMA) is run by its whole
// warp instead, with the lane-0-only instructions predicated: a lone lane
// executing while the other 31 wait at a warp or CTA barrier runs several
// times slower.  Every lane polls; the warp leaves when all lanes saw the
// phase complete, or, uniformly, when the wait gives up (bounded).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, 20000u))) return true;
    int give_up = 0;
    if ((threadIdx.x & 31) == 0) {
      give_up = *abort ? 1 : 0;
      if (!give_up && clock64() - t0 > kWaitBudgetCycles) {
        report(status, kDevTimeout);
        *abort = 1;
        give_up = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}

// ---------------------------------------------------------------- grid barrier
// All CTAs of the grid meet here.  The arrival counter only grows within a
// launch (it is cleared before the launch): barrier number k completes when
// it reaches k * gridDim.x, so an arrival is one release-add and the wait is
// a poll of the same word, with no reset round trip.  Returns false when a CTA
// recorded an error (a wait that ran out, here or anywhere in the grid): the
// caller then leaves the kernel.  Every wait is bounded.
__device__ bool grid_barrier(const PersistParams& P, State& st, const Ctx& c) {
  fence_proxy_async_all();  // this thread's generic writes before later async-proxy (TMA) reads
  tc_fence_before();        // TMEM reads of this phase before the next phase's MMAs
  __syncthreads();
  if (threadIdx.x < 32) {  // warp 0, converged; lane 0 arrives and polls
    const int lane = threadIdx.x;
    if (lane == 0 && *abort_flag(c)) atomicExch(P.grid_abort, 1);
    st.gen += 1;
    const unsigned target = st.gen * gridDim.x;
    if (lane == 0) red_add_release(P.bar_count, 1u);
    const long long t0 = clock64();
    unsigned i = 0;
    while (true) {
      int state = 0;  // 1 released, 2 give up
      if (lane == 0) {
        if ((int)(ld_acquire(P.bar_count) - target) >= 0) {
          state = 1;
        } else if ((++i & 31u) == 0) {
          if (*(volatile int*)P.grid_abort) {
            state = 2;
          } else if (clock64() - t0 > kWaitBudgetCycles) {
            report(P.status, kDevTimeout);
            atomicExch(P.grid_abort, 1);
            state = 2;
          }
        }
      }
      if (__shfl_sync(0xffffffffu, state, 0)) break;
      __nanosleep(P.spin_ns);  // back off: pollers contend with the phase's own traffic
    }
    if (lane == 0) c.ctrl->flag = *(volatile int*)P.grid_abort;
    __syncwarp();
  }
  __syncthreads();
  tc_fence_after();
  fence_proxy_async_all();
  return *(volatile int*)&c.ctrl->flag == 0;
}

// ---------------------------------------------------------------- GEMM phases
struct Unit {
  int n_tile, tt, ks, kb_begin, n_it;
};

__device__ __forceinline__ Unit gemm_unit(const PersistParams& P, const PersistGemm& G, int u) {
  Unit x;
  x.n_tile = u % G.n_tiles;
  const int r = u / G.n_tiles;
  x.tt = r % P.tok_tiles;
  x.ks = r / P.tok_tiles;
  x.kb_begin = (int)((long)x.ks * G.kb_total / G.ksplit);
  const int kb_end = (int)((long)(x.ks + 1) * G.kb_total / G.ksplit);
  x.n_it = kb_end - x.kb_begin;
  return x;
}

// Issue the weight tiles of this CTA's first unit of GEMM gi at `layer` into
// the free pipeline stages (the shared memory they land in must not be in use
// by the phases that run until the GEMM starts).  Called by every thread.
__device__ void gemm_prefetch(const PersistParams& P, State& st, const Ctx& c, int gi, int layer) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  st.prefetched = 0;
  const PersistGemm& G = P.g[gi];
  const int n_units = G.n_tiles * P.tok_tiles * G.ksplit;
  if ((int)blockIdx.x < n_units) {
    const Unit x = gemm_unit(P, G, blockIdx.x);
    const int S = P.stages;
    const int pre = x.n_it < S ? x.n_it : S;
    const uint32_t bytes = kATile + (uint32_t)P.tok_tile * 128;
    const int row = layer * G.rows_per_layer + x.n_tile * 128;
    const uint64_t pol = policy_evict_first();
    int it = 0;
    for (; it < pre; ++it) {
      const uint32_t g = st.pit + it;
      const int s = g % S;
      if (!warp_wait(&c.ctrl->empty[s], ((g / S) & 1u) ^ 1u, abort_flag(c), P.status)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&c.ctrl->full[s], bytes);
        tma_load_2d(c.smem + (size_t)s * kATile, &P.w[gi], &c.ctrl->full[s], (x.kb_begin + it) * 64, row, pol);
      }
    }
    st.prefetched = it;
    st.pre_gi = gi;
    st.pre_layer = layer;
  }
  __syncwarp();
}

// All threads: pull every weight tile this CTA's units of GEMM gi at `layer`
// will read into L2, one 128-byte line (a weight row's 64 K values) per
// prefetch.  These go through the load/store path, not the TMA unit, so they
// never queue in front of a phase's own TMA loads and stores.
__device__ void l2_prefetch_gemm(const PersistParams& P, int gi, int layer) {
  const PersistGemm& G = P.g[gi];
  const int n_units = G.n_tiles * P.tok_tiles * G.ksplit;
  const size_t K = (size_t)G.kb_total * 64;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Unit x = gemm_unit(P, G, u);
    if (x.tt != 0) continue;  // the token tiles of one weight slab share it
    const char* base = reinterpret_cast<const char*>(
        P.wptr[gi] + ((size_t)layer * G.rows_per_layer + (size_t)x.n_tile * 128) * K + (size_t)x.kb_begin * 64);
    const int lines = 128 * x.n_it;
    for (int i = threadIdx.x; i < lines; i += kPT) {
      const int r = i / x.n_it, kb = i - r * x.n_it;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(base + (size_t)r * K * 2 + (size_t)kb * 128));
    }
  }
}

__device__ void gemm_phase(const PersistParams& P, State& st, const Ctx& c, int gi, int layer) {
  const PersistGemm& G = P.g[gi];
  const int n_units = G.n_tiles * P.tok_tiles * G.ksplit;
  const int TT = P.tok_tile;
  const int btile = TT * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smA = c.smem;
  const int S = P.stages;
  uint8_t* smB = c.smem + (size_t)S * kATile;
  const uint32_t bytes = kATile + (uint32_t)btile;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Unit x = gemm_unit(P, G, u);
    const int t0 = x.tt * TT;
    if (warp == 0) {
      // ---- TMA producer: the warp runs the loop, lane 0 issues
      const int row = layer * G.rows_per_layer + x.n_tile * 128;
      const uint64_t pol = policy_evict_first();
      int pre = 0;
      if (u == (int)blockIdx.x && st.pre_gi == gi && st.pre_layer == layer) pre = st.prefetched;
      st.prefetched = 0;
      st.pre_gi = -1;
      int it = 0;
      for (; it < x.n_it; ++it) {
        const uint32_t g = st.pit + it;
        const int s = g % S;
        const int kc = (x.kb_begin + it) * 64;
        if (it >= pre) {
          if (!warp_wait(&c.ctrl->empty[s], ((g / S) & 1u) ^ 1u, abort_flag(c), P.status)) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&c.ctrl->full[s], bytes);
            tma_load_2d(smA + (size_t)s * kATile, &P.w[gi], &c.ctrl->full[s], kc, row, pol);
          }
        }
        if (lane == 0) tma_load_2d_nohint(smB + (size_t)s * btile, &P.act[gi], &c.ctrl->full[s], kc, t0);
      }
      if (it < pre) it = pre;  // the weights of the prefetched stages were issued
      st.pit += it;
      __syncwarp();
    } else if (warp == 1) {
      // ---- MMA issuer: the warp runs the loop, lane 0 issues
      const uint32_t idesc = idesc_bf16(128, TT);
      for (int it = 0; it < x.n_it; ++it) {
        const uint32_t g = st.mit + it;
        const int s = g % S;
        if (!warp_wait(&c.ctrl->full[s], (g / S) & 1u, abort_flag(c), P.status)) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t ad = sdesc_sw128(smem_u32(smA + (size_t)s * kATile));
          const uint64_t bd = sdesc_sw128(smem_u32(smB + (size_t)s * btile));
#pragma unroll
          for (int k = 0; k < 4; ++k) mma_bf16(c.tmem, ad + 2 * k, bd + 2 * k, idesc, (it > 0 || k > 0) ? 1u : 0u);
          mma_commit(&c.ctrl->empty[s]);
        }
        __syncwarp();
      }
      if (lane == 0) mma_commit(&c.ctrl->tmem_full);
      st.mit += x.n_it;
      st.units += 1;  // commits to tmem_full so far
      __syncwarp();
    } else if (warp >= 4) {
      // ---- epilogue: TMEM -> swizzled staging in the drained stages -> TMA stores
      const int q = warp & 3;
      const int n = x.n_tile * 128 + 32 * q + lane;
      const int ok = warp_wait(&c.ctrl->tmem_full, st.units & 1u, abort_flag(c), P.status) ? 1 : 0;
      st.units += 1;
      tc_fence_after();
      uint8_t* stg = c.smem;
      const uint32_t trow = (uint32_t)(32 * q) << 16;
      if (G.e_mode == kEPartial) {
        // warp q owns one box: [TT tokens][32 fp32] of output features 32q..32q+31
        uint8_t* box = stg + (size_t)q * TT * 128;
        const uint32_t lo = (uint32_t)((lane & 3) << 2);
        for (int c0 = 0; c0 < TT; c0 += 16) {
          float v[16];
          tmem_ld16(c.tmem + trow + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c0 + j;
            *reinterpret_cast<float*>(box + t * 128 + (((lane >> 2) ^ (t & 7)) << 4) + lo) = v[j];
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && ok) {
          tma_store_3d(&P.out[gi], box, x.n_tile * 128 + 32 * q, t0, x.ks);
          bulk_commit();
          bulk_wait_all();
        }
        __syncwarp();
      } else if (G.e_mode == kEQkvRope && G.tma_out) {
        // two boxes [TT tokens][64 bf16]: first and second members of the tile's 64 pairs
        const int half = P.dh >> 1;
        const int n0 = x.n_tile * 128;
        const int hb = n0 / P.dh;
        const int pair0 = (n0 - hb * P.dh) >> 1;
        const int p = n - hb * P.dh;
        const int pair = p >> 1, odd = p & 1;
        const int pl = pair - pair0;
        const bool rot = hb < P.n_rot_heads;
        uint8_t* box = stg + (size_t)odd * TT * 128;
        const uint32_t lo = (uint32_t)((pl & 7) << 1);
        for (int c0 = 0; c0 < TT; c0 += 16) {
          float2 csv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = t0 + c0 + j;
            csv[j] = (rot && t < P.M) ? __ldg(P.rope_cs + (size_t)t * half + pair) : make_float2(1.f, 0.f);
          }
          float v[16];
          tmem_ld16(c.tmem + trow + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            const int t = c0 + j;
            float outv = v[j];
            if (rot) {
              const float x1 = odd ? other : v[j], x2 = odd ? v[j] : other;
              outv = odd ? (x2 * csv[j].x + x1 * csv[j].y) : (x1 * csv[j].x - x2 * csv[j].y);
            }
            *reinterpret_cast<bf16*>(box + t * 128 + (((pl >> 3) ^ (t & 7)) << 4) + lo) = __float2bfloat16_rn(outv);
          }
        }
        fence_proxy_async_smem();
        named_bar(1, 128);
        if (threadIdx.x == 128 && ok) {
          tma_store_2d(&P.out[gi], stg, hb * P.dh + pair0, t0);
          tma_store_2d(&P.out[gi], stg + (size_t)TT * 128, hb * P.dh + half + pair0, t0);
          bulk_commit();
          bulk_wait_all();
        }
        __syncwarp();
      } else if (G.e_mode == kEQkvRope) {
        // head_dim 64: a 128-row tile spans two heads; direct stores
        const int half = P.dh >> 1;
        const int hb = n / P.dh, p = n - hb * P.dh;
        const int pair = p >> 1, odd = p & 1;
        const bool rot = hb < P.n_rot_heads;
        for (int c0 = 0; c0 < TT; c0 += 16) {
          float v[16];
          tmem_ld16(c.tmem + trow + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            const int t = t0 + c0 + j;
            if (t < P.M && ok) {
              float outv = v[j];
              if (rot) {
                const float2 cs = __ldg(P.rope_cs + (size_t)t * half + pair);
                const float x1 = odd ? other : v[j], x2 = odd ? v[j] : other;
                outv = odd ? (x2 * cs.x + x1 * cs.y) : (x1 * cs.x - x2 * cs.y);
              }
              P.qkv[(size_t)t * P.qkvdim + hb * P.dh + pair + odd * half] = __float2bfloat16_rn(outv);
            }
          }
        }
      } else {  // kEGeglu: one box [TT tokens][64 bf16] of GeGLU outputs n/2
        const int jl = 16 * q + (lane >> 1);
        const uint32_t lo = (uint32_t)((jl & 7) << 1);
        for (int c0 = 0; c0 < TT; c0 += 16) {
          float v[16];
          tmem_ld16(c.tmem + trow + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            const int t = c0 + j;
            if (!(lane & 1))
              *reinterpret_cast<bf16*>(stg + t * 128 + (((jl >> 3) ^ (t & 7)) << 4) + lo) =
                  __float2bfloat16_rn(gelu_tanh(v[j]) * other);
          }
        }
        fence_proxy_async_smem();
        named_bar(1, 128);
        if (threadIdx.x == 128 && ok) {
          tma_store_2d(&P.out[gi], stg, x.n_tile * 64, t0);
          bulk_commit();
          bulk_wait_all();
        }
        __syncwarp();
      }
    }
    tc_fence_before();
    __syncthreads();  // unit done: TMEM, stages and staging are free
    tc_fence_after();
  }
}

// ---------------------------------------------------------------- attention phase
// The tensor-core attention of the per-kernel path (heads of a KV group folded
// into 128-row query tiles, 64-key chunks of [valid prefix || actions], online
// softmax in the log2 domain, split-KV partials) run by warps 4..7: thread
// 128 + r owns query row r and TMEM lane r.  Warps 0..3 idle until the barrier.
__device__ __forceinline__ int fold_rows(int H) { return (H + 15) & ~15; }

// Gather code of key `j` of the chunk starting at key0 of request b: >= 0 a
// physical prefix row, -1 - i action row i, kSkip zero-fill (past the end).
__device__ __forceinline__ int chunk_code(const PersistParams& P, int b, int n_pre, int nk, int key0, int j) {
  const int key = key0 + j;
  if (j >= nk) return kSkip;
  if (key >= n_pre) return -1 - (key - n_pre);
  const int prow = P.valid_idx[(size_t)b * P.max_rows + key];
  if (prow >= 0 && prow < P.total_rows) return prow;
  report(P.status, kDevBounds);
  return kSkip;
}

struct AttnUnit {
  int b, g, qt, c_begin, c_end, n_pre, n_keys;
};

__device__ __forceinline__ AttnUnit attn_unit(const PersistParams& P, int u) {
  AttnUnit a;
  const int sp = u % P.max_splits;
  u /= P.max_splits;
  a.qt = u % P.q_tiles;
  u /= P.q_tiles;
  a.g = u % P.Hkv;
  a.b = u / P.Hkv;
  a.n_pre = P.n_valid[a.b];
  a.n_keys = a.n_pre + P.H;
  const int n_chunks = (a.n_keys + kChunk - 1) / kChunk;
  a.c_begin = sp * P.chunks_per_cta;
  a.c_end = min(a.c_begin + P.chunks_per_cta, n_chunks);
  return a;
}

// Once per launch, all threads: the gather codes of every chunk this CTA's
// attention units visit, in visiting order, if they fit the cache.
__device__ void attn_codes_init(const PersistParams& P, const Ctx& c) {
  const int n_units = P.batch * P.Hkv * P.q_tiles * P.max_splits;
  int total = 0;
  for (int u0 = blockIdx.x; u0 < n_units; u0 += gridDim.x) {
    const AttnUnit a = attn_unit(P, u0);
    if (a.c_begin < a.c_end) total += a.c_end - a.c_begin;
  }
  if (total > kCodeChunks) {
    if (threadIdx.x == 0) c.ctrl->n_cached = -1;
    return;
  }
  int slot = 0;
  for (int u0 = blockIdx.x; u0 < n_units; u0 += gridDim.x) {
    const AttnUnit a = attn_unit(P, u0);
    for (int cc = a.c_begin; cc < a.c_end; ++cc, ++slot) {
      const int key0 = cc * kChunk;
      const int nk = min(kChunk, a.n_keys - key0);
      for (int j = threadIdx.x; j < kChunk; j += kPT) c.ctrl->codes[slot][j] = chunk_code(P, a.b, a.n_pre, nk, key0, j);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int sl = 0; sl < total; ++sl) {
      const int* ix = c.ctrl->codes[sl];
      // codes increase strictly over a chunk's prefix keys: first and last decide
      c.ctrl->slot_row[sl] = (ix[0] >= 0 && ix[kChunk - 1] >= 0 && ix[kChunk - 1] - ix[0] == kChunk - 1) ? ix[0] : -1;
    }
    c.ctrl->n_cached = total;
  }
}

// Warp 4 (attention thread 0 issues): start the K/V loads of this CTA's first
// attention chunk of `layer` when it is a TMA chunk (prefix rows do not depend
// on the phases before attention), and pull the CTA's other TMA chunks into L2.
// The shared memory it lands in must be free.
__device__ void attn_prefetch(const PersistParams& P, State& st, const Ctx& c, int layer) {
  if ((threadIdx.x >> 5) != 4) return;
  const int lane = threadIdx.x & 31;
  if (c.ctrl->n_cached > 0) {
    const int dh = P.dh, kdb = dh / 64;
    const uint32_t kvb = (uint32_t)dh * kChunk * 2;
    uint8_t* K0 = c.smem + (uint32_t)dh * 256;
    uint8_t* V0 = K0 + 2 * kvb;
    const int n_units = P.batch * P.Hkv * P.q_tiles * P.max_splits;
    const int layer_row0 = layer * (int)P.total_rows;
    int slot = 0;
    for (int u0 = blockIdx.x; u0 < n_units; u0 += gridDim.x) {
      const AttnUnit a = attn_unit(P, u0);
      for (int cc = a.c_begin; cc < a.c_end; ++cc, ++slot) {
        const int r0 = c.ctrl->slot_row[slot];
        if (r0 < 0) continue;
        if (slot == 0) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&c.ctrl->bar_kv[0], 2u * kdb * kChunk * 128);
            for (int kb = 0; kb < kdb; ++kb) {
              tma_load_2d_nohint(K0 + kb * kChunk * 128, &P.pk, &c.ctrl->bar_kv[0], a.g * dh + kb * 64, layer_row0 + r0);
              tma_load_2d_nohint(V0 + kb * kChunk * 128, &P.pv, &c.ctrl->bar_kv[0], a.g * dh + kb * 64, layer_row0 + r0);
            }
          }
          st.kv_pend[0] = 1;
          st.kv_pre = 1;
        } else if (lane < kdb) {
          tma_prefetch_l2_2d(&P.pk, a.g * dh + lane * 64, layer_row0 + r0);
          tma_prefetch_l2_2d(&P.pv, a.g * dh + lane * 64, layer_row0 + r0);
        }
      }
    }
  }
  __syncwarp();
}

__device__ void attn_phase(const PersistParams& P, State& st, const Ctx& c, int layer) {
  if (threadIdx.x < 128) return;
  const int at = threadIdx.x - 128;
  const int w = at >> 5, lane = at & 31;
  const int dh = P.dh;
  const int kdb = dh / 64;
  const int G = P.Hq / P.Hkv;
  const int Hp = fold_rows(P.H);
  const int n_units = P.batch * P.Hkv * P.q_tiles * P.max_splits;
  const uint32_t kvb = (uint32_t)dh * kChunk * 2;
  uint8_t* Q = c.smem;
  uint8_t* Kb[2] = {Q + (uint32_t)dh * 256, Q + (uint32_t)dh * 256 + kvb};
  uint8_t* Vb[2] = {Q + (uint32_t)dh * 256 + 2 * kvb, Q + (uint32_t)dh * 256 + 3 * kvb};
  uint8_t* Pm = Q + (uint32_t)dh * 256 + 4 * kvb;
  Ctrl* k = c.ctrl;
  const uint32_t tm_o = c.tmem, tm_s = c.tmem + (uint32_t)dh;
  const uint32_t lane_off = (uint32_t)(32 * w) << 16;
  const int layer_row0 = layer * (int)P.total_rows;
  const int kvdim = P.Hkv * dh;
  const bf16* pk = P.pk_ptr + (size_t)layer_row0 * kvdim;
  const bf16* pv = P.pv_ptr + (size_t)layer_row0 * kvdim;
  const float sl2 = P.scale * kLog2e;
  const bool cached = k->n_cached >= 0;
  int next_slot = 0;

  for (int u0 = blockIdx.x; u0 < n_units; u0 += gridDim.x) {
    int u = u0;
    const int sp = u % P.max_splits;
    u /= P.max_splits;
    const int qt = u % P.q_tiles;
    u /= P.q_tiles;
    const int g = u % P.Hkv;
    const int b = u / P.Hkv;
    const int n_pre = P.n_valid[b];
    const int n_keys = n_pre + P.H;
    const int n_chunks = (n_keys + kChunk - 1) / kChunk;
    const int c_begin = sp * P.chunks_per_cta;
    const int c_end = min(c_begin + P.chunks_per_cta, n_chunks);
    if (c_begin >= c_end) continue;  // uniform for the 128 threads
    const int n_my = c_end - c_begin;
    const int slot0 = next_slot;
    next_slot += n_my;

    // codes of chunk cc into buffer bf (>= 0 prefix row, -1 - i action row i,
    // kSkip zero-fill); a contiguous run of 64 prefix rows arrives by TMA,
    // anything else is gathered row by row with cp.async
    auto load_chunk = [&](int cc, int bf, int slot) -> bool {
      const int* ix;
      bool contiguous;
      if (cached) {
        ix = k->codes[slot];
        contiguous = k->slot_row[slot] >= 0;
      } else {
        const int key0 = cc * kChunk;
        const int nk = min(kChunk, n_keys - key0);
        int* wx = k->idx[bf];
        if (at < kChunk) wx[at] = chunk_code(P, b, n_pre, nk, key0, at);
        named_bar(2, 128);
        ix = wx;
        contiguous = nk == kChunk && ix[0] >= 0 && ix[kChunk - 1] - ix[0] == kChunk - 1;
      }
      if (contiguous) {
        if (w == 0 && !(st.kv_pre && slot == 0)) {
          if (lane == 0) mbar_arrive_expect_tx(&k->bar_kv[bf], 2u * kdb * kChunk * 128);
          const int row = layer_row0 + ix[0];
          if (lane == 0)
            for (int kb = 0; kb < kdb; ++kb) {
              tma_load_2d_nohint(Kb[bf] + kb * kChunk * 128, &P.pk, &k->bar_kv[bf], g * dh + kb * 64, row);
              tma_load_2d_nohint(Vb[bf] + kb * kChunk * 128, &P.pv, &k->bar_kv[bf], g * dh + kb * 64, row);
            }
          st.kv_pend[bf] = 1;
        }
        if (w == 0) st.kv_pre = 0;
        __syncwarp();
      } else {
        const int cpr = dh / 8;                    // 16-byte pieces per row
        const int rpw = cpr >= 32 ? 1 : 32 / cpr;  // rows per warp instruction
        const int ppl = cpr >= 32 ? cpr / 32 : 1;  // pieces per lane per row
        const int sub = lane / (32 / rpw), pl = lane % (32 / rpw);
        for (int j0 = w * rpw; j0 < kChunk; j0 += 4 * rpw) {
          const int j = j0 + sub;
          const int code = ix[j];
          const bf16* kr = P.qkv;  // any valid address when zero-filling
          const bf16* vr = P.qkv;
          uint32_t nbytes = 0;
          if (code >= 0) {
            kr = pk + (size_t)code * kvdim + g * dh;
            vr = pv + (size_t)code * kvdim + g * dh;
            nbytes = 16;
          } else if (code != kSkip) {
            const bf16* base = P.qkv + (size_t)(b * P.H + (-1 - code)) * P.qkvdim;
            kr = base + (P.Hq + g) * dh;
            vr = base + (P.Hq + P.Hkv + g) * dh;
            nbytes = 16;
          }
          for (int e = 0; e < ppl; ++e) {
            const int ch = pl + e * 32;
            const uint32_t off = (ch >> 3) * kChunk * 128 + sw128_offset(j, ch & 7);
            cp_async16(Kb[bf] + off, nbytes ? kr + ch * 8 : kr, nbytes);
            cp_async16(Vb[bf] + off, nbytes ? vr + ch * 8 : vr, nbytes);
          }
        }
        cp_async_commit();
      }
      return contiguous;
    };

    bool tma_cur = load_chunk(c_begin, 0, slot0);
    // query tile by TMA: 16-row groups of the fold (a group never straddles heads)
    if (w == 0) {
      int nbox = 0;
      for (int rg = 0; rg < 8; ++rg)
        if ((qt * 128 + rg * 16) / Hp < G) ++nbox;
      if (lane == 0) mbar_arrive_expect_tx(&k->bar_q, (uint32_t)nbox * kdb * 16 * 128);
      for (int rg = 0; rg < 8 && lane == 0; ++rg) {
        const int r0 = qt * 128 + rg * 16;
        const int hh = r0 / Hp;
        if (hh >= G) continue;
        const int tok0 = r0 - hh * Hp;
        for (int kb = 0; kb < kdb; ++kb)
          tma_load_2d_nohint(Q + kb * 128 * 128 + rg * 16 * 128, &P.q16, &k->bar_q, (g * G + hh) * dh + kb * 64,
                             b * P.H + tok0);
      }
      st.q_pend = 1;
    }
    __syncwarp();
    float m_ref = -INFINITY, l = 0.f;
    const int row = at;
    for (int ci = 0; ci < n_my; ++ci) {
      const int cc = c_begin + ci;
      const int bf = ci & 1;
      const int nk = min(kChunk, n_keys - cc * kChunk);
      bool tma_next = false;
      const bool has_next = ci + 1 < n_my;
      if (has_next) tma_next = load_chunk(cc + 1, bf ^ 1, slot0 + ci + 1);
      if (!tma_cur) {
        if (has_next && !tma_next) cp_async_wait<1>();
        else cp_async_wait<0>();
        fence_proxy_async_smem();
      }
      if (w == 0) {
        if (tma_cur) {
          warp_wait(&k->bar_kv[bf], st.kv_ph[bf], abort_flag(c), P.status);
          st.kv_ph[bf] ^= 1u;
          st.kv_pend[bf] = 0;
        }
        if (ci == 0) {
          warp_wait(&k->bar_q, st.q_uses & 1u, abort_flag(c), P.status);
          st.q_pend = 0;
        }
      }
      __syncwarp();
      tc_fence_before();
      named_bar(2, 128);
      tc_fence_after();
      // ---- S = Q K^T
      if (at == 0) {
        const uint32_t idesc = idesc_bf16(128, kChunk);
        for (int kb = 0; kb < kdb; ++kb) {
          const uint64_t ad = sdesc_sw128(smem_u32(Q + kb * 128 * 128));
          const uint64_t bd = sdesc_sw128(smem_u32(Kb[bf] + kb * kChunk * 128));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tm_s, ad + 2 * kk, bd + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&k->bar_s);
      }
      __syncwarp();
      warp_wait(&k->bar_s, st.s_uses & 1u, abort_flag(c), P.status);
      tc_fence_after();
      float s[kChunk];
      tmem_ld64(tm_s + lane_off, s);
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        s[j] *= sl2;
        if (j < nk) mx[j & 3] = fmaxf(mx[j & 3], s[j]);
      }
      const float cmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      float factor = 1.f;
      if (ci == 0) {
        m_ref = cmax;
      } else if (cmax > m_ref + kRescaleMargin * kLog2e) {
        factor = ex2_fast(m_ref - cmax);
        m_ref = cmax;
      }
      if (__any_sync(0xffffffffu, factor != 1.f)) {
        l *= factor;
#pragma unroll 1
        for (int c0 = 0; c0 < dh; c0 += 16) {
          float v[16];
          tmem_ld16(tm_o + lane_off + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] *= factor;
          tmem_st16(tm_o + lane_off + (uint32_t)c0, v);
        }
      }
      uint32_t pk2[kChunk / 2];
#pragma unroll
      for (int j = 0; j < kChunk; j += 2) {
        const float p0 = (j < nk) ? ex2_fast(s[j] - m_ref) : 0.f;
        const float p1 = (j + 1 < nk) ? ex2_fast(s[j + 1] - m_ref) : 0.f;
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
        const float2 pr = __bfloat1622float2(pb);  // the row sum uses the weights P V multiplies
        l += pr.x + pr.y;
        pk2[j / 2] = *reinterpret_cast<const uint32_t*>(&pb);
      }
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8)
        *reinterpret_cast<uint4*>(Pm + sw128_offset(row, q8)) =
            make_uint4(pk2[4 * q8], pk2[4 * q8 + 1], pk2[4 * q8 + 2], pk2[4 * q8 + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar(2, 128);
      tc_fence_after();
      // ---- O += P V (V is the MN-major operand)
      if (at == 0) {
        const uint32_t idesc = idesc_bf16(128, dh, true);
        const uint64_t ad = sdesc_sw128(smem_u32(Pm));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = sdesc_sw128_mn(smem_u32(Vb[bf] + kk * 2048), kChunk * 128, 1024);
          mma_bf16(tm_o, ad + 2 * kk, bd, idesc, (ci > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&k->bar_o);
      }
      __syncwarp();
      warp_wait(&k->bar_o, st.s_uses & 1u, abort_flag(c), P.status);
      tc_fence_after();
      st.s_uses += 1;
      tma_cur = tma_next;
    }
    st.q_uses += 1;
    cp_async_wait<0>();
    named_bar(2, 128);  // every chunk buffer is free: stage O in the K/V space
    // O rows -> swizzled staging boxes of 32 fp32 columns x 128 rows -> TMA stores
    const int r = qt * 128 + row;
    const bool valid_row = r / Hp < G && r % Hp < P.H;
    uint8_t* stg = Kb[0];
    for (int c0 = 0; c0 < dh; c0 += 64) {
      float v[64];
      tmem_ld64(tm_o + lane_off + (uint32_t)c0, v);
#pragma unroll
      for (int q4 = 0; q4 < 16; ++q4) {
        const int col = c0 + 4 * q4;
        uint8_t* box = stg + (col >> 5) * (128 * 128);
        *reinterpret_cast<float4*>(box + sw128_offset(row, (col & 31) >> 2)) =
            make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
      }
    }
    if (valid_row) P.attn_ml[(size_t)u0 * 128 + row] = make_float2(m_ref, l);
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(2, 128);
    if (at == 0) {
      for (int bx = 0; bx < dh / 32; ++bx) tma_store_2d(&P.attn_o, stg + bx * (128 * 128), bx * 32, u0 * 128);
      bulk_commit();
      bulk_wait_all();
    }
    __syncwarp();
    named_bar(2, 128);
    tc_fence_after();
  }
}

// ---------------------------------------------------------------- row and element phases
// These phases are short and latency-bound: every thread issues all of its
// independent loads before it consumes any, so a phase costs about one or two
// L2 round trips instead of one per split.
__device__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  __syncthreads();  // red is free (a previous use has been read)
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kPT / 32; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

// h = x W_in^T + b_in of token row t, then the first layer's adaRMS.
// W_in rows are A bf16 long; with A % 8 == 0 a thread reads 4 rows as 16-byte
// vectors, 4 vectors of each at a time, before it multiplies.
__device__ void inproj_phase(const PersistParams& P, const Ctx& c, int step) {
  const float* mod = P.mod + ((size_t)step * P.L * 2) * 3 * P.D;
  float* xs = c.rows;
  const int A = P.A, D = P.D, A8 = P.A / 8;
  const bool vec = (A & 7) == 0;
  for (int t = blockIdx.x; t < P.M; t += gridDim.x) {
    __syncthreads();
    for (int k = threadIdx.x; k < A; k += kPT) xs[k] = P.x[(size_t)t * A + k];
    __syncthreads();
    float* hr = P.h + (size_t)t * D;
    float* dump = P.dump ? P.dump + (((size_t)step * (P.L + 1)) * P.M + t) * D : nullptr;
    float ss = 0.f;
    for (int n0 = threadIdx.x; n0 < D; n0 += 4 * kPT) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (vec) {
        for (int kb = 0; kb < A8; kb += 4) {
          uint4 q[4][4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int n = n0 + e * kPT;
              q[e][j] = (n < D && kb + j < A8) ? __ldg(reinterpret_cast<const uint4*>(P.w_in + (size_t)n * A) + kb + j)
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
          const int n = n0 + e * kPT;
          if (n < D)
            for (int k = 0; k < A; ++k) acc[e] += xs[k] * __bfloat162float(P.w_in[(size_t)n * A + k]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = n0 + e * kPT;
        if (n >= D) continue;
        const float hn = acc[e] + __bfloat162float(P.b_in[n]);
        hr[n] = hn;
        ss += hn * hn;
        if (dump) dump[n] = hn;
      }
    }
    ss = block_sum(ss, c.ctrl->red);
    const float r = 1.0f / sqrtf(ss / (float)D + P.eps);
    for (int n = threadIdx.x; n < D; n += kPT)
      P.y[(size_t)t * D + n] = __float2bfloat16_rn(hr[n] * r * (1.f + mod[n]) + mod[D + n]);
  }
}

// Token row t: h += gate * (sum of the split-K partials in split order); then,
// if `mod` is given, y = adaRMS(h) with (scale, shift) = (mod, mod + D).
// A thread owns up to 4 columns and loads 8 splits of all of them at once.
__device__ void resid_norm_phase(const PersistParams& P, const Ctx& c, const float* part, int ks_n,
                                 const float* gate, const float* mod, float* dump_base) {
  const int D = P.D;
  const size_t stride = (size_t)P.M * D;
  constexpr int kCols = 4, kSplitBlock = 8;
  for (int t = blockIdx.x; t < P.M; t += gridDim.x) {
    float* hr = P.h + (size_t)t * D;
    float ss = 0.f;
    for (int n0 = threadIdx.x; n0 < D; n0 += kPT * kCols) {
      float acc[kCols];
      bool in[kCols];
#pragma unroll
      for (int e = 0; e < kCols; ++e) {
        acc[e] = 0.f;
        in[e] = n0 + e * kPT < D;
      }
      const float* pp = part + (size_t)t * D + n0;
      for (int j0 = 0; j0 < ks_n; j0 += kSplitBlock) {
        float v[kSplitBlock][kCols];
#pragma unroll
        for (int jj = 0; jj < kSplitBlock; ++jj)
#pragma unroll
          for (int e = 0; e < kCols; ++e)
            v[jj][e] = (j0 + jj < ks_n && in[e]) ? __ldcg(pp + (size_t)(j0 + jj) * stride + e * kPT) : 0.f;
#pragma unroll
        for (int jj = 0; jj < kSplitBlock; ++jj)
#pragma unroll
          for (int e = 0; e < kCols; ++e)
            if (j0 + jj < ks_n) acc[e] += v[jj][e];
      }
#pragma unroll
      for (int e = 0; e < kCols; ++e) {
        if (!in[e]) continue;
        const int n = n0 + e * kPT;
        const float hn = hr[n] + gate[n] * acc[e];
        hr[n] = hn;
        ss += hn * hn;
        if (dump_base) dump_base[(size_t)t * D + n] = hn;
      }
    }
    if (mod == nullptr) continue;
    ss = block_sum(ss, c.ctrl->red);
    const float r = 1.0f / sqrtf(ss / (float)D + P.eps);
    for (int n = threadIdx.x; n < D; n += kPT)
      P.y[(size_t)t * D + n] = __float2bfloat16_rn(hr[n] * r * (1.f + mod[n]) + mod[D + n]);
  }
}

// Split-K sum of the merged QKV projection in split order, RoPE on q and k.
__device__ void reduce_qkv_phase(const PersistParams& P, const float* part, int ks_n) {
  const int N = P.qkvdim, np = N >> 1, half = P.dh >> 1;
  const long total = (long)P.M * np;
  for (long idx = (long)blockIdx.x * kPT + threadIdx.x; idx < total; idx += (long)gridDim.x * kPT) {
    const int t = (int)(idx / np), pp = (int)(idx - (long)t * np);
    const int n = 2 * pp;
    float x1 = 0.f, x2 = 0.f;
    for (int j0 = 0; j0 < ks_n; j0 += 8) {
      float2 v[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        v[jj] = j0 + jj < ks_n ? __ldcg(reinterpret_cast<const float2*>(part + ((size_t)(j0 + jj) * P.M + t) * N + n))
                               : make_float2(0.f, 0.f);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (j0 + jj < ks_n) {
          x1 += v[jj].x;
          x2 += v[jj].y;
        }
    }
    const int hb = n / P.dh, pair = (n - hb * P.dh) >> 1;
    float o1 = x1, o2 = x2;
    if (hb < P.n_rot_heads) {
      const float2 cs = P.rope_cs[(size_t)t * half + pair];
      o1 = x1 * cs.x - x2 * cs.y;
      o2 = x2 * cs.x + x1 * cs.y;
    }
    P.qkv[(size_t)t * N + hb * P.dh + pair] = __float2bfloat16_rn(o1);
    P.qkv[(size_t)t * N + hb * P.dh + pair + half] = __float2bfloat16_rn(o2);
  }
}

// GeGLU of the split-K partials of the interleaved gate/up projection.
__device__ void geglu_reduce_phase(const PersistParams& P, const float* part, int ks_n) {
  const int F = P.F;
  const long total = (long)P.M * F;
  for (long idx = (long)blockIdx.x * kPT + threadIdx.x; idx < total; idx += (long)gridDim.x * kPT) {
    const int t = (int)(idx / F), j = (int)(idx - (long)t * F);
    float g = 0.f, u = 0.f;
    for (int s0 = 0; s0 < ks_n; s0 += 8) {
      float2 v[8];
#pragma unroll
      for (int ss = 0; ss < 8; ++ss)
        v[ss] = s0 + ss < ks_n
                    ? __ldcg(reinterpret_cast<const float2*>(part + ((size_t)(s0 + ss) * P.M + t) * 2 * F + 2 * j))
                    : make_float2(0.f, 0.f);
#pragma unroll
      for (int ss = 0; ss < 8; ++ss)
        if (s0 + ss < ks_n) {
          g += v[ss].x;
          u += v[ss].y;
        }
    }
    P.m[idx] = __float2bfloat16_rn(gelu_tanh(g) * u);
  }
}

// Merge the chunk ranges of every query row in range order; bf16 o[token][head dh + d].
// dh / 4 threads per row (one float4 of the partial each), kPT * 4 / dh rows per pass.
__device__ void combine_phase(const PersistParams& P) {
  const int G = P.Hq / P.Hkv, Hp = fold_rows(P.H);
  const int rows = P.batch * P.Hq * P.H;
  const int tpr = P.dh / 4;
  const int rpp = kPT / tpr;
  const int d4 = threadIdx.x % tpr;
  constexpr int kSp = 16;
  for (int R = blockIdx.x * rpp + threadIdx.x / tpr; R < rows; R += gridDim.x * rpp) {
    const int b = R / (P.Hq * P.H);
    const int rr = R - b * P.Hq * P.H;
    const int g = rr / (G * P.H), hr = rr % (G * P.H);
    const int hh = hr / P.H, tok = hr % P.H;
    const int r = hh * Hp + tok;
    const int qt = r / 128, row = r % 128;
    const int n_chunks = (P.n_valid[b] + P.H + kChunk - 1) / kChunk;
    const int n_splits = (n_chunks + P.chunks_per_cta - 1) / P.chunks_per_cta;
    const size_t unit0 = ((size_t)((b * P.Hkv + g) * P.q_tiles + qt)) * P.max_splits;
    float m = -INFINITY;
    for (int s0 = 0; s0 < n_splits; s0 += kSp) {
      float mv[kSp];
#pragma unroll
      for (int j = 0; j < kSp; ++j)
        mv[j] = s0 + j < n_splits ? __ldcg(&P.attn_ml[(unit0 + s0 + j) * 128 + row].x) : -INFINITY;
#pragma unroll
      for (int j = 0; j < kSp; ++j) m = fmaxf(m, mv[j]);
    }
    float l = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n_splits; s0 += kSp) {
      float2 ml[kSp];
      float4 ov[kSp];
#pragma unroll
      for (int j = 0; j < kSp; ++j) {
        const bool in = s0 + j < n_splits;
        const size_t u = unit0 + s0 + j;
        ml[j] = in ? __ldcg(&P.attn_ml[u * 128 + row]) : make_float2(-INFINITY, 0.f);
        ov[j] = in ? __ldcg(reinterpret_cast<const float4*>(P.attn_o_ptr + (u * 128 + row) * P.dh) + d4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kSp; ++j) {
        if (s0 + j >= n_splits) continue;
        const float wgt = ex2_fast(ml[j].x - m);
        l += ml[j].y * wgt;
        acc.x += ov[j].x * wgt;
        acc.y += ov[j].y * wgt;
        acc.z += ov[j].z * wgt;
        acc.w += ov[j].w * wgt;
      }
    }
    const int h = g * G + hh;
    __nv_bfloat162* dst =
        reinterpret_cast<__nv_bfloat162*>(P.o + (size_t)(b * P.H + tok) * (P.Hq * P.dh) + h * P.dh + 4 * d4);
    dst[0] = __floats2bfloat162_rn(acc.x / l, acc.y / l);
    dst[1] = __floats2bfloat162_rn(acc.z / l, acc.w / l);
  }
}

// Final adaRMS (scale, shift), action output projection, x += delta * v.
__device__ void final_phase(const PersistParams& P, const Ctx& c, int step) {
  float* yf = c.rows;
  const int D = P.D;
  const float* fin = P.fin + (size_t)step * 2 * D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < P.M; t += gridDim.x) {
    const float* hr = P.h + (size_t)t * D;
    float ss = 0.f;
    for (int k = threadIdx.x; k < D; k += kPT) ss += hr[k] * hr[k];
    ss = block_sum(ss, c.ctrl->red);
    const float r = 1.0f / sqrtf(ss / (float)D + P.eps);
    for (int k = threadIdx.x; k < D; k += kPT) yf[k] = hr[k] * r * (1.f + fin[k]) + fin[D + k];
    __syncthreads();
    // warp w: outputs w, w + 8, w + 16, w + 24 together; a lane reads 16-byte
    // vectors k8 = lane + 32 j of each output's W_out row
    const int D8 = D / 8;
    for (int a0 = warp; a0 < P.A; a0 += 4 * (kPT / 32)) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k0 = lane; k0 < D8; k0 += 4 * 32) {
        uint4 q[4][4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int a = a0 + e * (kPT / 32), k8 = k0 + 32 * j;
            q[e][j] = (a < P.A && k8 < D8) ? __ldg(reinterpret_cast<const uint4*>(P.w_out + (size_t)a * D) + k8)
                                           : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int k8 = k0 + 32 * j;
            if (k8 >= D8) continue;
            float f[8];
            bf16x8_to_f32(q[e][j], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[e] += yf[8 * k8 + i] * f[i];
          }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int a = a0 + e * (kPT / 32);
        const float sum = warp_sum(v[e]);
        if (lane == 0 && a < P.A) P.x[(size_t)t * P.A + a] += P.delta * (sum + __bfloat162float(P.b_out[a]));
      }
    }
    __syncthreads();
  }
}

// All threads of the grid: bring a table into L2 (one prefetch per 128-byte line).
__device__ void l2_warm(const void* p, size_t bytes) {
  const char* b = static_cast<const char*>(p);
  for (size_t off = ((size_t)blockIdx.x * kPT + threadIdx.x) * 128; off < bytes; off += (size_t)gridDim.x * kPT * 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(b + off));
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kPT, 1) k_persistent(const __grid_constant__ PersistParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Ctx c;
  c.smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // keeps the shared address space
  c.rows = reinterpret_cast<float*>(c.smem + P.data_bytes);
  c.ctrl = reinterpret_cast<Ctrl*>(c.smem + P.data_bytes + P.row_bytes);
  const int warp = threadIdx.x >> 5;
  State st;
  st.gen = 0;
  st.pit = st.mit = st.units = 0;
  st.pre_gi = -1;
  st.pre_layer = -1;
  st.prefetched = 0;
  st.q_uses = st.s_uses = 0;
  st.kv_ph[0] = st.kv_ph[1] = 0;
  st.kv_pend[0] = st.kv_pend[1] = st.q_pend = 0;
  st.kv_pre = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&c.ctrl->full[s], 1);
      mbar_init(&c.ctrl->empty[s], 1);
    }
    mbar_init(&c.ctrl->tmem_full, 1);
    mbar_init(&c.ctrl->bar_s, 1);
    mbar_init(&c.ctrl->bar_o, 1);
    mbar_init(&c.ctrl->bar_q, 1);
    mbar_init(&c.ctrl->bar_kv[0], 1);
    mbar_init(&c.ctrl->bar_kv[1], 1);
    c.ctrl->abort = 0;
    c.ctrl->flag = 0;
    fence_mbar_init();
    for (int i = 0; i < 4; ++i) {
      prefetch_tensormap(&P.w[i]);
      prefetch_tensormap(&P.act[i]);
      if (P.g[i].tma_out) prefetch_tensormap(&P.out[i]);
    }
    prefetch_tensormap(&P.q16);
    prefetch_tensormap(&P.attn_o);
    if (P.total_rows >= kChunk) {
      prefetch_tensormap(&P.pk);
      prefetch_tensormap(&P.pv);
    }
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(&c.ctrl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = c.ctrl->tmem_base;
  attn_codes_init(P, c);
  __syncthreads();
  // the small tables every phase reads: modulation, final modulation, W_in, W_out
  l2_warm(P.mod, (size_t)P.n_steps * P.L * 2 * 3 * P.D * sizeof(float));
  l2_warm(P.fin, (size_t)P.n_steps * 2 * P.D * sizeof(float));
  l2_warm(P.w_in, (size_t)P.D * P.A * sizeof(bf16));
  l2_warm(P.w_out, (size_t)P.A * P.D * sizeof(bf16));

  const int L = P.L, D = P.D;
  bool alive = true;
  for (int step = 0; step < P.n_steps && alive; ++step) {
    if (step == 0) {
      if (P.l2_pf) l2_prefetch_gemm(P, 0, 0);
      gemm_prefetch(P, st, c, 0, 0);
    }
    inproj_phase(P, c, step);
    if (!(alive = grid_barrier(P, st, c))) break;
    for (int l = 0; l < L; ++l) {
      const float* mod1 = P.mod + (((size_t)step * L + l) * 2 + 0) * 3 * D;
      const float* mod2 = mod1 + 3 * D;
      // merged QKV (+ RoPE); then this CTA's first prefix K/V chunk
      gemm_phase(P, st, c, 0, l);
      attn_prefetch(P, st, c, l);
      if (!(alive = grid_barrier(P, st, c))) break;
      if (P.g[0].ksplit > 1) {
        reduce_qkv_phase(P, P.part0, P.g[0].ksplit);
        if (!(alive = grid_barrier(P, st, c))) break;
      }
      // attention over [valid prefix || actions], then the O weights
      attn_phase(P, st, c, l);
      __syncthreads();
      gemm_prefetch(P, st, c, 1, l);
      if (!(alive = grid_barrier(P, st, c))) break;
      if (P.l2_pf) l2_prefetch_gemm(P, 2, l);
      combine_phase(P);
      if (!(alive = grid_barrier(P, st, c))) break;
      // O projection -> gated residual -> adaRMS2
      gemm_phase(P, st, c, 1, l);
      gemm_prefetch(P, st, c, 2, l);
      if (!(alive = grid_barrier(P, st, c))) break;
      if (P.l2_pf) l2_prefetch_gemm(P, 3, l);
      if (P.l2_pf) l2_prefetch_gemm(P, 0, (l + 1) % L);
      resid_norm_phase(P, c, P.part0, P.g[1].ksplit, mod1 + 2 * D, mod2, nullptr);
      if (!(alive = grid_barrier(P, st, c))) break;
      // merged gate/up (+ GeGLU)
      gemm_phase(P, st, c, 2, l);
      gemm_prefetch(P, st, c, 3, l);
      if (!(alive = grid_barrier(P, st, c))) break;
      if (P.g[2].ksplit > 1) {
        geglu_reduce_phase(P, P.part0, P.g[2].ksplit);
        if (!(alive = grid_barrier(P, st, c))) break;
      }
      // down projection -> gated residual -> adaRMS1 of the next layer
      gemm_phase(P, st, c, 3, l);
      const bool more = l + 1 < L || step + 1 < P.n_steps;
      if (more) gemm_prefetch(P, st, c, 0, (l + 1) % L);
      if (!(alive = grid_barrier(P, st, c))) break;
      const float* nxt = l + 1 < L ? P.mod + (((size_t)step * L + l + 1) * 2) * 3 * D : nullptr;
      float* dump = P.dump ? P.dump + (((size_t)step * (L + 1) + l + 1) * P.M) * D : nullptr;
      if (P.l2_pf) l2_prefetch_gemm(P, 1, (l + 1) % L);
      resid_norm_phase(P, c, P.part1, P.g[3].ksplit, mod2 + 2 * D, nxt, dump);
      if (!(alive = grid_barrier(P, st, c))) break;
    }
    if (!alive) break;
    final_phase(P, c, step);
    if (!(alive = grid_barrier(P, st, c))) break;
  }

  // Leave with nothing in flight: stores, gathers, TMA loads and MMAs.
  cp_async_wait<0>();
  if (warp == 0) {
    if (threadIdx.x == 0) {
      bulk_wait_all();
      // the last phase issued on each stage (a weight prefetch may be unconsumed)
      volatile int fresh = 0;
      const uint32_t total = st.pit + (uint32_t)st.prefetched;
      const uint32_t S = (uint32_t)P.stages;
      for (uint32_t g = total > S ? total - S : 0; g < total; ++g)
        mbar_wait(&c.ctrl->full[g % S], (g / S) & 1u, &fresh, P.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (threadIdx.x == 32 && !alive) {
      // MMAs of an interrupted unit complete before TMEM is freed: one more
      // commit, then phases units - 1 and units of tmem_full in order
      volatile int fresh = 0;
      mma_commit(&c.ctrl->tmem_full);
      if (st.units > 0) mbar_wait(&c.ctrl->tmem_full, (st.units - 1) & 1u, &fresh, P.status);
      mbar_wait(&c.ctrl->tmem_full, st.units & 1u, &fresh, P.status);
    }
    __syncwarp();
  } else if (warp == 4) {
    if (threadIdx.x == 128) {
      bulk_wait_all();
      volatile int fresh = 0;
      if (st.q_pend) mbar_wait(&c.ctrl->bar_q, st.q_uses & 1u, &fresh, P.status);
      for (int b = 0; b < 2; ++b)
        if (st.kv_pend[b]) mbar_wait(&c.ctrl->bar_kv[b], st.kv_ph[b], &fresh, P.status);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(c.tmem, 512);
  }
}

}  // namespace

// Dynamic shared memory of the persistent kernel: the data region holds the
// larger of the GEMM pipeline (stages x (weight tile + token tile)) and the
// attention tiles; then the row scratch and the control block.  The pipeline
// gets as many stages (up to 8) as fit the shared memory left by the rest.
size_t persist_smem_bytes(int tok_tile, int dh, int D, int A, uint32_t* data_bytes, uint32_t* row_bytes,
                          int* stages) {
  const size_t stage = kATile + (size_t)tok_tile * 128;
  const size_t attn = (size_t)dh * 256 + 4 * (size_t)dh * kChunk * 2 + 128 * kChunk * 2;
  size_t r = (size_t)(D > A ? D : A) * sizeof(float);
  r = (r + 127) & ~(size_t)127;
  const size_t budget = (232448 - 1024 - r - sizeof(Ctrl)) & ~(size_t)1023;
  int S = (int)(budget / stage);
  if (S > kMaxStages) S = kMaxStages;
  if (S < 4) S = 4;
  size_t d = (size_t)S * stage > attn ? (size_t)S * stage : attn;
  d = (d + 1023) & ~(size_t)1023;
  if (data_bytes) *data_bytes = (uint32_t)d;
  if (row_bytes) *row_bytes = (uint32_t)r;
  if (stages) *stages = S;
  return 1024 + d + r + sizeof(Ctrl);
}

cudaError_t persist_setup(size_t smem, int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(k_persistent, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_persistent, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_persistent, kPT, smem);
  return e;
}

cudaError_t launch_persistent(const PersistParams& P, int grid, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once, or the launch fails
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_persistent, P);
}

}  // namespace ae
