// dec_attention_noalloc: the split-KV decode attention kernel for callers that
// must not allocate device memory.  Its scratch (the per-CTA partial records,
// the per-head arrival counters, the step position and the error flag) lives
// in one file-scope __device__ array instead of a cudaMalloc'd workspace.
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <mutex>

#include "../../include/dec.h"
#include "common.cuh"
#include "kernels.h"

using namespace tld;

namespace {

// Limits of the fixed scratch.
constexpr int kNoAllocRecordFloats = 1 << 18;  // 1 MiB of partial records
constexpr int kNoAllocMaxKvHeads = 64;
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocScratch {
  float records[kNoAllocRecordFloats];
  int counters[kNoAllocMaxKvHeads];
  int pos;
  int err;
  int err_line;  // first failing source line of a debug build's index check
};

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) NoAllocScratch g_noalloc_scratch;

// Per-device set-up, done once by the first call on each device.  `done` is
// published with release order after the other fields are written, so a thread
// that reads it true (acquire) sees them; the mutex keeps two first callers on
// one device from both running the set-up.
struct DeviceSetup {
  std::atomic<bool> done{false};
  NoAllocScratch* scratch = nullptr;  // device address of g_noalloc_scratch
  int n_sm = 0;
};
DeviceSetup g_setup[kNoAllocMaxDevices];
std::mutex g_setup_mutex[kNoAllocMaxDevices];

// The device address of the scratch array and the SM count, with device `dev`
// current.  Nothing here allocates.
int setup_device(int dev, DeviceSetup& su) {
  if (su.done.load(std::memory_order_acquire)) return DEC_OK;
  std::lock_guard<std::mutex> lock(g_setup_mutex[dev]);
  if (su.done.load(std::memory_order_relaxed)) return DEC_OK;
  // The host-side symbol is only a stand-in: the kernels need the device address.
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return DEC_ERR_CUDA;
  int n_sm = 0;
  if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DEC_ERR_CUDA;
  if (set_smem_limits() != cudaSuccess) return DEC_ERR_CUDA;
  su.scratch = static_cast<NoAllocScratch*>(ptr);
  su.n_sm = n_sm;
  su.done.store(true, std::memory_order_release);
  return DEC_OK;
}

// Clears the counters and the error flag and stores the position of this call.
__global__ void noalloc_prepare(NoAllocScratch* s, int pos, int n_counters) {
  for (int i = threadIdx.x; i < n_counters; i += blockDim.x) s->counters[i] = 0;
  if (threadIdx.x == 0) {
    s->pos = pos;
    s->err = 0;
    s->err_line = 0;
  }
}

}  // namespace

extern "C" int dec_attention_noalloc(const float* q, const void* k_cache, const void* v_cache,
                                     int n_q_heads, int n_kv_heads, int head_dim, int ctx_stride,
                                     int n, float* o, dec_stream_t stream) {
  if (!q || !k_cache || !v_cache || !o) return DEC_ERR_ARG;
  if (head_dim != 64 && head_dim != 128) return DEC_ERR_SHAPE;
  if (n_kv_heads < 1 || n_kv_heads > kNoAllocMaxKvHeads || n_q_heads < 1 ||
      n_q_heads % n_kv_heads)
    return DEC_ERR_SHAPE;
  const int G = n_q_heads / n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return DEC_ERR_SHAPE;
  if (ctx_stride < 1 || ctx_stride > 65536 || n < 1 || n > ctx_stride) return DEC_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return DEC_ERR_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return DEC_ERR_CUDA;
  DeviceSetup& su = g_setup[dev];
  if (setup_device(dev, su) != DEC_OK) return DEC_ERR_CUDA;

  // Same grid and ring as the decoder's attention launch.
  const int grid = su.n_sm < (kMaxSplits - 1) * n_kv_heads ? su.n_sm : (kMaxSplits - 1) * n_kv_heads;
  if ((size_t)grid * 2 * G * (head_dim + 4) > (size_t)kNoAllocRecordFloats) return DEC_ERR_SHAPE;
  const size_t fixed = attn_smem_bytes(head_dim, G, 0);
  int ns = (int)(((size_t)kSmemBudget > fixed ? kSmemBudget - fixed : 0) / kAttnStageBytes);
  ns = ns < 2 ? 2 : (ns > 6 ? 6 : ns);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  {
    // launched through cudaLaunchKernelExC so that only this launch's own error
    // is seen (an earlier, unrelated error of the caller stays pending)
    NoAllocScratch* scratch = su.scratch;
    int pos = n - 1, n_counters = n_kv_heads;
    void* args[] = {&scratch, &pos, &n_counters};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(64);
    cfg.stream = s;
    if (cudaLaunchKernelExC(&cfg, (const void*)noalloc_prepare, args) != cudaSuccess)
      return DEC_ERR_CUDA;
  }

  AttnParams p{};
  p.kc = static_cast<const uint16_t*>(k_cache);
  p.vc = static_cast<const uint16_t*>(v_cache);
  p.q = q;
  p.o = o;
  p.part = su.scratch->records;
  p.counters = su.scratch->counters;
  p.pos = &su.scratch->pos;
  p.err = &su.scratch->err;
  p.nkv = n_kv_heads;
  p.max_ctx = ctx_stride;
  p.nstages = ns;
  p.scale = (float)(1.0 / std::sqrt((double)head_dim));
  p.tl = nullptr;
  if (launch_attn(head_dim, G, p, grid, attn_smem_bytes(head_dim, G, ns), s, false) != cudaSuccess)
    return DEC_ERR_CUDA;
  return DEC_OK;
}

namespace tld {

// The error flag of the no-alloc attention kernel on the current device, read
// after `stream` has drained, then cleared (dec_sync_status with a NULL
// handle).  cudaMemcpyFromSymbol / ToSymbol allocate nothing.  Returns DEC_OK,
// DEC_ERR_DEVICE (flag was set) or DEC_ERR_CUDA.
int noalloc_sync_status(cudaStream_t stream, int* flag_out) {
  *flag_out = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return DEC_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DEC_ERR_CUDA;
  if (!g_setup[dev].done.load(std::memory_order_acquire)) return DEC_OK;  // never called here
  int flag = 0;
  if (cudaMemcpyFromSymbol(&flag, g_noalloc_scratch, sizeof(int),
                           offsetof(NoAllocScratch, err)) != cudaSuccess)
    return DEC_ERR_CUDA;
  if (flag == 0) return DEC_OK;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(int), offsetof(NoAllocScratch, err)) !=
      cudaSuccess)
    return DEC_ERR_CUDA;
  *flag_out = flag;
  return DEC_ERR_DEVICE;
}

}  // namespace tld
