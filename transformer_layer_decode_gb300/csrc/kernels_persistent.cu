// The persistent per-token kernel: one cooperative launch runs every layer of
// a decode step, one CTA per SM.  Its phases are the fused layer's five
// (norm + QKV + RoPE + append, attention, o-proj + residual, norm + gate/up +
// SwiGLU, down + residual), separated by grid-wide barriers instead of kernel
// boundaries.  The producer thread streams the whole step's bytes - for each
// layer this CTA's QKV slab, its K/V chunks, then its o, gate/up and down slabs
// - through one shared-memory ring without stopping at phase ends, so HBM keeps
// streaming the next phase while the consumers finish the current one and
// wait at the barrier.  Only the K/V chunk that holds this step's appended row
// waits for the QKV phase of its layer.
#include "phases.cuh"

namespace tld {

namespace {

// Grid barrier of the consumers: every CTA arrives once per phase; phase k of
// the step is complete when the counter reaches (k + 1) * gridDim.x.
__device__ __forceinline__ void grid_arrive(int* ctr, int tid) {
  named_barrier(1, kNC);  // this CTA's writes of the phase are done
  if (tid == 0) {
    __threadfence();
    atomicAdd(ctr, 1);
  }
}

__device__ __forceinline__ void grid_wait(const int* ctr, int target, int* err, int tid,
                                          uint64_t* tl) {
  if (tid == 0) {
    spin_until(ctr, target, err);
    __threadfence();
    tl_mark_min(tl, 0);
    tl_mark_max(tl, 1);
  }
  named_barrier(1, kNC);
}

// Timeline slots of phase k: P.tl + kTimelineSlots * k.
__device__ __forceinline__ uint64_t* phase_tl(const TokenParams& P, int k) {
  return P.tl ? P.tl + (size_t)kTimelineSlots * k : nullptr;
}

// State the consumers carry from phase to phase.
struct PhaseCtx {
  uint8_t* work;
  Ring R;
  RingPos cp;
  int* ctr;
  int* err;
  int tid, b, nb;
};

// One GEMV phase of one layer.  The parameter block is copied into locals, so
// that its inner loop reads registers rather than memory its own stores could
// alias.
template <int PRO, int EPI, bool Q4>
__device__ __forceinline__ bool gemv_phase(const GemvParams& pin, const GemvIO& io, PhaseCtx& cx,
                                           int target, uint64_t* tl) {
  const GemvParams p = pin;
  const int tid = cx.tid;
  const int rb0 = (int)split_begin(p.n_rb, cx.nb, cx.b);
  const int rb1 = (int)split_begin(p.n_rb, cx.nb, cx.b + 1);
  const GemvWork W(cx.work, GemvLayout{p.geo.K, p.max_rb_local, Q4});
  gemv_pre<PRO>(p, io.norm_w, W, tid);  // norm weights do not depend on the previous phase
  if (target > 0) grid_wait(cx.ctr, target, cx.err, tid, tl);
  const bool ok = gemv_main<PRO, EPI, Q4>(p, io, W, cx.R, cx.cp, rb0, rb1, tid, cx.b == 0);
  if (tid == 0) {
    tl_mark_min(tl, 2);
    tl_mark_max(tl, 3);
  }
  grid_arrive(cx.ctr, tid);
  return ok;
}

template <int HD, int G>
__device__ __forceinline__ bool attn_phase(const AttnParams& pin, int pos, int att_grid,
                                           PhaseCtx& cx, int target, uint64_t* tl) {
  const AttnParams p = pin;
  AttnSplit S = attn_split<HD>(pos, p.nkv, cx.b < att_grid ? cx.b : 0, att_grid);
  if (cx.b >= att_grid) S.u0 = S.u1 = S.U, S.nu = 0;
  const int tid = cx.tid;
  grid_wait(cx.ctr, target, cx.err, tid, tl);
  const bool ok = attn_main<HD, G>(p, cx.work, cx.R, cx.cp, S, cx.b, att_grid, tid);
  if (tid == 0) {
    tl_mark_min(tl, 2);
    tl_mark_max(tl, 3);
  }
  grid_arrive(cx.ctr, tid);
  return ok;
}

// GEMV inputs and outputs of layer l's GEMV `slot` (kernel id `kernel`): the
// int8 input taps and the block-dot tap are set when the caller asked for them.
__device__ __forceinline__ GemvIO gemv_io(const TokenParams& P, int l, int slot, int kernel,
                                          const uint8_t* w, const uint16_t* norm_w,
                                          const float* x, float* x_copy, float* out, float* tap,
                                          uint16_t* kc, uint16_t* vc) {
  GemvIO io{w, norm_w, x, x_copy, out, tap, kc, vc, nullptr, nullptr, nullptr};
  if (P.qtap) {
    io.qtap = P.qtap + ((size_t)l * 4 + slot) * P.km;
    io.qstap = P.qstap + ((size_t)l * 4 + slot) * (P.km / 32);
  }
  if (P.dots && P.dot_layer == l && P.dot_kernel == kernel) io.dots = P.dots;
  return io;
}

// The five phases of one layer, inlined into the layer loop.  With five phases
// in one loop body the compiler keeps values of several phases live at once and
// spills about a kilobyte per thread (a non-inlined layer or phase function
// spills as much and runs slower still), where each standalone fused kernel
// spills nothing.  That is why this plan's phases run slower than the
// five-kernel plan's kernels.
template <int HD, int G, bool Q4>
__device__ __forceinline__ bool layer_phases(const TokenParams* Pp, int l, int pos, PhaseCtx* cxp) {
  const TokenParams& Q = *Pp;
  PhaseCtx cx = *cxp;
  const int nb = cx.nb, k0 = 5 * l, L = Q.n_layers;
  bool ok = true;
  {
    const PLayer& ly = Q.layers[l];
    const GemvIO io = gemv_io(Q, l, 0, 0, ly.wqkv, ly.attn_norm, l == 0 ? Q.emb : Q.X,
                              l == 0 ? Q.X : nullptr, nullptr, nullptr, ly.kc, ly.vc);
    ok &= gemv_phase<PRO_NORM, EPI_QKV, Q4>(Q.qkv, io, cx, k0 * nb, phase_tl(Q, k0));
  }
  ok &= attn_phase<HD, G>(Q.attn, pos, Q.att_grid, cx, (k0 + 1) * nb, phase_tl(Q, k0 + 1));
  {
    const GemvIO io = gemv_io(Q, l, 1, 2, Q.layers[l].wo, nullptr, Q.o.x, nullptr, Q.o.out,
                              nullptr, nullptr, nullptr);
    ok &= gemv_phase<PRO_PLAIN, EPI_RESID, Q4>(Q.o, io, cx, (k0 + 2) * nb, phase_tl(Q, k0 + 2));
  }
  {
    const PLayer& ly = Q.layers[l];
    const GemvIO io = gemv_io(Q, l, 2, 3, ly.wgu, ly.ffn_norm, Q.gu.x, nullptr, nullptr, nullptr,
                              nullptr, nullptr);
    ok &= gemv_phase<PRO_NORM, EPI_SWIGLU, Q4>(Q.gu, io, cx, (k0 + 3) * nb, phase_tl(Q, k0 + 3));
  }
  {
    const GemvIO io = gemv_io(Q, l, 3, 4, Q.layers[l].wd, nullptr, Q.down.x, nullptr,
                              l == L - 1 ? Q.out : Q.X,
                              Q.tap ? Q.tap + (size_t)l * Q.hidden : nullptr, nullptr, nullptr);
    ok &= gemv_phase<PRO_PLAIN, EPI_RESID, Q4>(Q.down, io, cx, (k0 + 4) * nb, phase_tl(Q, k0 + 4));
  }
  cxp->cp = cx.cp;
  return ok;
}

}  // namespace

template <int HD, int G, bool Q4>
__global__ void __launch_bounds__(kThreads, 1) token_persistent(const __grid_constant__ TokenParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Ring R{smem, reinterpret_cast<uint64_t*>(smem + (size_t)P.nstages * P.slot_bytes),
               reinterpret_cast<uint64_t*>(smem + (size_t)P.nstages * P.slot_bytes) + P.nstages,
               P.nstages, P.slot_bytes};
  uint8_t* work = smem + (size_t)P.nstages * P.slot_bytes + 16 * (size_t)P.nstages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  const int L = P.n_layers;
  // The step position and the barrier counter of this step (two counters
  // alternate by position parity; the other one belongs to the previous step,
  // which has finished, and is cleared here for the next).
  const int pos = *P.pos;
  int* ctr = P.bar + (pos & 1);
  if (b == 0 && tid == 0) P.bar[(pos & 1) ^ 1] = 0;

  if (tid == 0) {
    ring_init(R);
    tl_mark_min(phase_tl(P, 0), 5);
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      AttnSplit S = attn_split<HD>(pos, P.attn.nkv, b < P.att_grid ? b : 0, P.att_grid);
      if (b >= P.att_grid) S.u0 = S.u1 = S.U, S.nu = 0;  // CTAs past the attention grid idle there
      RingPos RP{0, 0, 0};
      auto rb = [&](const GemvParams& m, int i) { return (int)split_begin(m.n_rb, nb, b + i); };
#pragma unroll 1
      for (int l = 0; l < L; ++l) {
        const PLayer ly = P.layers[l];
        gemv_produce(P.qkv, ly.wqkv, R, RP, rb(P.qkv, 0), rb(P.qkv, 1), pol);
        attn_produce<HD>(P.attn, ly.kc, ly.vc, R, RP, S, pol, [&] {
          // the appended row was written by other CTAs' QKV epilogues
          spin_until(ctr, (5 * l + 1) * nb, P.err);
          fence_proxy_async_global();
        });
        gemv_produce(P.o, ly.wo, R, RP, rb(P.o, 0), rb(P.o, 1), pol);
        gemv_produce(P.gu, ly.wgu, R, RP, rb(P.gu, 0), rb(P.gu, 1), pol);
        gemv_produce(P.down, ly.wd, R, RP, rb(P.down, 0), rb(P.down, 1), pol);
      }
    }
    return;
  }

  PhaseCtx cx{work, R, RingPos{0, 0, 0}, ctr, P.err, tid, b, nb};
  bool ok = true;
#pragma unroll 1
  for (int l = 0; l < L; ++l) ok &= layer_phases<HD, G, Q4>(&P, l, pos, &cx);
  // the step is over when every CTA has finished the last phase
  grid_wait(ctr, 5 * L * nb, P.err, tid, nullptr);
  if (b == 0 && tid == 0) atomicAdd(P.pos, 1);
  if (!ok && tid == 0) ring_drain(R, cx.cp, P.err);
}

size_t persistent_work_bytes(const TokenParams& P, int hd, int G, bool q4) {
  size_t w = AttnLayout{hd, G}.total();
  for (const GemvParams* m : {&P.qkv, &P.o, &P.gu, &P.down}) {
    const size_t g = GemvLayout{m->geo.K, m->max_rb_local, q4}.total();
    if (g > w) w = g;
  }
  return (w + 127) & ~(size_t)127;
}

const void* persistent_kernel_ptr(int hd, int G, bool q4) {
#define TLD_P(H_, G_)                                                               \
  if (hd == H_ && G == G_)                                                          \
    return q4 ? (const void*)token_persistent<H_, G_, true>                         \
              : (const void*)token_persistent<H_, G_, false>;
  TLD_P(64, 1) TLD_P(64, 2) TLD_P(64, 4) TLD_P(64, 8)
  TLD_P(128, 1) TLD_P(128, 2) TLD_P(128, 4) TLD_P(128, 8)
#undef TLD_P
  return nullptr;
}

cudaError_t launch_persistent(int hd, int G, bool q4, const TokenParams& P, int grid, size_t smem,
                              cudaStream_t s) {
  const void* fn = persistent_kernel_ptr(hd, G, q4);
  if (!fn) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  TokenParams copy = P;
  void* args[] = {&copy};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: grid barriers are safe
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace tld
