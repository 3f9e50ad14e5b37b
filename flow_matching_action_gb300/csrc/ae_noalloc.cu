// ae_sample_noalloc: ae_sample for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc at sampling time: code running while a
// stream capture is open (allocation would invalidate the capture), code whose
// device memory comes from a fixed budget owned by someone else (a serving
// process that pre-reserves HBM for its KV caches), or real-time control loops
// that forbid allocator calls after start-up.  ae_sample may allocate on its
// first use of a new n_steps (the time-conditioning table) and when it captures
// its CUDA graph.  This entry point runs the same kernels, launched directly on
// the context's stream, and allocates nothing: the split-KV partial results of
// the attention kernel live in one file-scope __device__ array of fixed size
// instead of in context memory.
#include <mutex>

#include "ae_internal.h"

namespace {

// 16 MiB of attention partials, held by every GPU that loads this library
// until the process exits.
constexpr size_t kScratchFloats = (size_t)4 << 20;
static __device__ __align__(256) float g_attn_scratch[kScratchFloats];

// Device address of g_attn_scratch per device.  In host code the symbol's name
// is only a host-side stand-in, so the address is looked up with that device
// current and passed to the kernels as a plain pointer.  It is cached per
// device together with the CUDA context it was looked up in: after
// cudaDeviceReset the device gets a new primary context, in which the module
// (and the array) is loaded again, so a lookup from another context is redone.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (CtxGetCurrentFn)p;
  }
  return fn;
}

cudaError_t scratch_address(int device, float** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return e;
  if (cur != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
  CUcontext ctx = nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr || get(&ctx) != CUDA_SUCCESS) e = cudaErrorNotSupported;
  if (e == cudaSuccess && (g_scratch_addr[device] == nullptr || g_scratch_ctx[device] != ctx)) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e == cudaSuccess) {
      g_scratch_addr[device] = static_cast<float*>(p);
      g_scratch_ctx[device] = ctx;
    }
  }
  if (cur != device) cudaSetDevice(cur);
  if (e != cudaSuccess) return e;
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

void set_msg(ae_ctx* c, const char* m) { c->last_msg = m; }

}  // namespace

extern "C" ae_status ae_sample_noalloc(ae_ctx* c, const float* noise, int n_steps, float* out) {
  if (c == nullptr) return AE_ERR_INVALID_ARG;
  if (!c->fast) {
    set_msg(c, "ae_sample_noalloc needs a bf16 context (AE_DTYPE_BF16)");
    return AE_ERR_UNSUPPORTED;
  }
  if (c->bind.batch < 0) {
    set_msg(c, "ae_sample_noalloc before ae_bind_prefix");
    return AE_ERR_NOT_BOUND;
  }
  if (n_steps < 1 || n_steps > AE_MAX_STEPS) {
    set_msg(c, "n_steps outside 1..AE_MAX_STEPS");
    return AE_ERR_SHAPE;
  }
  const int B = c->bind.batch;
  if (B > 0 && (noise == nullptr || out == nullptr)) {
    set_msg(c, "noise / out_actions is NULL");
    return AE_ERR_INVALID_ARG;
  }
  if (c->status_host && *(volatile int*)c->status_host != 0) {
    set_msg(c, "a device-side check failed earlier");
    return AE_ERR_DEVICE;
  }
  const ae::Dims& d = c->d;
  if (c->dump != nullptr &&
      (size_t)n_steps * (d.L + 1) * B * d.H * d.D > c->dump_cap) {
    set_msg(c, "debug dump too small for this sample");
    return AE_ERR_SHAPE;
  }
  c->launches_sample = 0;
  if (B == 0) return AE_OK;
  // building a time table allocates: it must come from an earlier ae_sample
  const ae::TimeTable* t = ae::find_time_table(c, n_steps);
  if (t == nullptr) {
    set_msg(c, "no time-conditioning table for this n_steps yet: call ae_sample once with the same "
               "n_steps (it builds and caches the table) before ae_sample_noalloc");
    return AE_ERR_NOT_BOUND;
  }
  // the attention partials of this batch must fit the fixed scratch
  ae::AttnScratch sc;
  const size_t per_unit = (size_t)128 * d.dh + 2 * 128;  // O rows + (max, sum) pairs
  sc.max_units = (int)(kScratchFloats / per_unit);
  ae::AttnArgs probe = {};
  probe.batch = B;
  probe.H = d.H;
  probe.Hq = d.Hq;
  probe.Hkv = d.Hkv;
  probe.dh = d.dh;
  probe.plan_rows = c->bind.max_phys_rows;
  probe.max_units = sc.max_units;
  const size_t units = ae::attn_plan_units(probe, c->sm_count);
  if (units > (size_t)sc.max_units) {
    set_msg(c, "batch too large for the fixed 16 MiB attention scratch of ae_sample_noalloc "
               "(it holds one 128-row query tile per request and KV head at least)");
    return AE_ERR_SHAPE;
  }
  float* base = nullptr;
  cudaError_t e = scratch_address(c->device, &base);
  if (e != cudaSuccess) {
    c->last_msg = std::string("cudaGetSymbolAddress of the static scratch: ") + cudaGetErrorString(e);
    return AE_ERR_CUDA;
  }
  sc.part_o = base;
  sc.part_ml = reinterpret_cast<float2*>(base + (size_t)sc.max_units * 128 * d.dh);
  e = ae::make_attn_o_map(&sc.omap, sc.part_o, (size_t)sc.max_units, d.dh);  // host-side encode only
  if (e != cudaSuccess) {
    c->last_msg = std::string("TMA descriptor of the static scratch: ") + cudaGetErrorString(e);
    return AE_ERR_CUDA;
  }

  const size_t xbytes = (size_t)B * d.H * d.A * sizeof(float);
  if (out != noise) {
    e = cudaMemcpyAsync(out, noise, xbytes, cudaMemcpyDeviceToDevice, c->stream);
    if (e != cudaSuccess) {
      c->last_msg = std::string("copy of the noise: ") + cudaGetErrorString(e);
      return AE_ERR_CUDA;
    }
  }
  int64_t n = 0;
  for (int s = 0; s < n_steps; ++s) {
    n += ae::launch_step_fast(c, *t, s, out, c->stream, &e, &sc);
    if (e != cudaSuccess) {
      c->last_msg = std::string("bf16 step launch: ") + cudaGetErrorString(e);
      return AE_ERR_CUDA;
    }
  }
  c->launches_sample = n;
  return AE_OK;
}
