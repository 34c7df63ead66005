// Fused decode-layer kernels for sm_103a.
//
// Five kernels per layer (the fusions of "RDNA4 Decode Kernel Fusion:
// Pipeline Barriers, Not Launches, Are the Win", FAQ and section "Fusion
// removes the barrier by removing the write"):
//   K1 gemv<PRO_NORM,  EPI_QKV>    RMSNorm*w, [Wq;Wk;Wv] GEMV, RoPE on q and k
//                                  and the k/v append in the epilogue
//   K2 attn_decode                 GQA split-KV attention: one thread-block
//                                  cluster per KV head, merged in distributed
//                                  shared memory (or a flat grid whose split
//                                  heads the last CTA of each merges)
//   K3 gemv<PRO_PLAIN, EPI_RESID>  Wo GEMV + residual add
//   K4 gemv<PRO_NORM,  EPI_SWIGLU> RMSNorm*w, interleaved gate/up GEMV,
//                                  silu(g)*u in the epilogue (g, u never stored)
//   K5 gemv<PRO_PLAIN, EPI_RESID>  Wd GEMV + residual add
//
// Batch-1 projections are matrix-vector products: one flop per weight byte, so
// they are bound by HBM, not by the tensor cores.  Each GEMV CTA owns a
// contiguous run of whole 4-row blocks of the tiled weight matrix, i.e. one
// contiguous slab of bytes, and streams it through a ring of 32 KB
// shared-memory stages filled by 1-D bulk copies (TMA) issued by one producer
// thread.  Sixteen consumer warps each take one 4-row tile per stage (256
// columns bf16, 1024 int4), copy it to registers, hand the stage back, and
// accumulate against the input vector held in shared memory in fp32.  Because
// CTAs own whole rows, no partial sums cross CTAs.  Weights do not depend on
// the previous kernel: the producer starts streaming at launch, before
// griddepcontrol.wait.
#include "phases.cuh"

namespace tld {

// Shared memory of a standalone phase kernel: ring | mbarriers | work area.
size_t gemv_smem_bytes(int K, bool q4, int nstages, int max_rb_local) {
  return (size_t)nstages * (q4 ? kStageBytesQ4 : kStageBytes) + 16 * (size_t)nstages +
         GemvLayout{K, max_rb_local, q4}.total();
}

// Consumer warps of the attention kernel: 16 for the cluster kernels of GQA
// groups up to 2 and of group 4 at head_dim 64 (their registers allow 17
// warps a CTA; at head_dim 64 a group of 4 needs 16 warps to keep the
// one-butterfly form), else 8 (measured: 16 warps slow group 4 at head_dim 128
// by 2 %, with or without a ring stage fewer).
constexpr int attn_warps(int hd, int G, bool cluster) {
  return cluster && (G <= 2 || (G == 4 && hd == 64)) ? 16 : kAttnWarps;
}
int attn_consumer_warps(int hd, int G, bool cluster) { return attn_warps(hd, G, cluster); }

size_t attn_smem_bytes(int hd, int G, int nstages, bool cluster) {
  return (size_t)nstages * kAttnStageBytes + 16 * (size_t)nstages +
         AttnLayout{hd, G, attn_consumer_warps(hd, G, cluster), cluster}.total();
}

template <int PRO, int EPI, bool Q4>
__global__ void __launch_bounds__(kThreads, 1) gemv_fused(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Ring R{smem, reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * p.geo.stage_bytes),
               reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * p.geo.stage_bytes) + p.nstages,
               p.nstages, p.geo.stage_bytes};
  uint8_t* work = smem + (size_t)p.nstages * p.geo.stage_bytes + 16 * (size_t)p.nstages;
  const GemvWork W(work, GemvLayout{p.geo.K, p.max_rb_local, Q4});
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  if (tid == 0) tl_mark_min(p.tl, 0);
  // whole row blocks [rb0, rb1) of this CTA
  const int rb0 = (int)split_begin(p.n_rb, nb, b), rb1 = (int)split_begin(p.n_rb, nb, b + 1);
  if (tid == 0) ring_init(R);
  __syncthreads();

  if (warp == kConsumerWarps) {
    // producer: weights only, so it streams before griddepcontrol.wait
    if (lane == 0) {
      RingPos P{0, 0, 0};
      gemv_produce(p, p.w, R, P, rb0, rb1, policy_evict_first());
      l2_ahead(p.ahead, b);
    }
    return;
  }
  gemv_pre<PRO>(p, p.norm_w, W, tid);
  pdl_wait();  // the input vector comes from the previous kernel
  if (tid == 0) {
    tl_mark_min(p.tl, 2);
    tl_mark_max(p.tl, 3);
  }
  // Let the next kernel launch (and start its weight stream) now.  Triggering
  // only after this CTA's own wait keeps at most two kernels in flight and means
  // everything before the previous kernel is complete when the next one starts.
  pdl_trigger();
  RingPos P{0, 0, 0};
  const bool ok = gemv_main<PRO, EPI, Q4>(p, gemv_io(p), W, R, P, rb0, rb1, tid, b == 0);
  if (!ok) {
    if (tid == 0) ring_drain(R, P, p.err);
    return;
  }
  if (p.tl) {
    named_barrier(1, kNC);
    if (tid == 0) {
      tl_mark_max(p.tl, 1);
      tl_mark_min(p.tl, 7);
    }
  }
}

template <int HD, int G, bool CL, int NW>
__global__ void __launch_bounds__((NW + 1) * 32, 1) attn_decode(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Ring R{smem, reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * kAttnStageBytes),
               reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * kAttnStageBytes) + p.nstages,
               p.nstages, kAttnStageBytes};
  uint8_t* work = smem + (size_t)p.nstages * kAttnStageBytes + 16 * (size_t)p.nstages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  if (tid == 0) tl_mark_min(p.tl, 0);
  // The step position is read before griddepcontrol.wait: it was last written by
  // the previous step's final kernel, and this kernel can only launch after the
  // preceding kernel's CTAs have all passed their own wait, i.e. after that
  // final kernel completed.
  const int pos = *p.pos;
  const AttnSplit S = CL ? attn_split_cluster<HD>(pos, p.nkv, b, p.cluster)
                         : attn_split<HD>(pos, p.nkv, b, nb);
  if (tid == 0) ring_init(R, NW);
  __syncthreads();
  // cluster: the CTAs push their records into each other's shared memory at
  // the end; this first cluster barrier phase (waited for before the first
  // push) makes sure every CTA of the cluster is running by then
  if (CL) cluster_arrive_relaxed();

  if (warp == NW) {
    if (lane == 0) {
      RingPos P{0, 0, 0};
      attn_produce<HD>(p, p.kc, p.vc, R, P, S, policy_evict_first(), [] { pdl_wait(); });
      l2_ahead(p.ahead, b);
    }
    if (CL) {  // the producer warp takes part in the consumers' two cluster barrier phases
      __syncwarp();
      cluster_wait();
      cluster_sync_all();
    }
    return;
  }
  pdl_wait();  // q comes from the QKV kernel
  pdl_trigger();
  if (tid == 0) {
    tl_mark_min(p.tl, 2);
    tl_mark_max(p.tl, 3);
  }
  RingPos P{0, 0, 0};
  const bool ok = attn_main<HD, G, CL, NW>(p, work, R, P, S, b, nb, tid);
  if (p.tl) {
    named_barrier(1, NW * 32);
    if (tid == 0) {
      tl_mark_max(p.tl, 1);
      tl_mark_min(p.tl, 7);
    }
  }
  if (!ok && tid == 0) ring_drain(R, P, p.err);
}

// ---- the LM head and the greedy token ------------------------------------------
// Order-preserving key of a logit at row j: the float's bits mapped so that
// unsigned order is float order, and the row's complement below them, so the
// largest key is the largest logit at its lowest row.
__device__ __forceinline__ unsigned long long argmax_key(float v, int j) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (uint32_t)~(uint32_t)j;
}

// Final RMSNorm x weight and the vocabulary GEMV (logits to p.g.out), then the
// greedy token: each CTA reduces its own rows' logits to one key, takes the
// maximum with the global key, and the last CTA to finish (a ticket) writes
// the token and clears the key and the ticket for the next launch.  The
// maximum does not depend on the order of arrival, so the token is the same
// every run.
__global__ void __launch_bounds__(kThreads, 1) lm_head_argmax(const LmHeadParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GemvParams& p = P.g;
  const Ring R{smem, reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * p.geo.stage_bytes),
               reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * p.geo.stage_bytes) + p.nstages,
               p.nstages, p.geo.stage_bytes};
  uint8_t* work = smem + (size_t)p.nstages * p.geo.stage_bytes + 16 * (size_t)p.nstages;
  const GemvWork W(work, GemvLayout{p.geo.K, p.max_rb_local, false});
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  const int rb0 = (int)split_begin(p.n_rb, nb, b), rb1 = (int)split_begin(p.n_rb, nb, b + 1);
  if (tid == 0) ring_init(R);
  __syncthreads();
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      RingPos Pp{0, 0, 0};
      gemv_produce(p, p.w, R, Pp, rb0, rb1, policy_evict_first());
    }
    return;
  }
  gemv_pre<PRO_NORM>(p, p.norm_w, W, tid);
  pdl_wait();  // the stack's output comes from the last layer
  pdl_trigger();
  RingPos Pp{0, 0, 0};
  const bool ok = gemv_main<PRO_NORM, EPI_LOGITS, false>(p, gemv_io(p), W, R, Pp, rb0, rb1, tid, b == 0);
  if (!ok) {
    if (tid == 0) ring_drain(R, Pp, p.err);
    return;
  }
  named_barrier(1, kNC);  // this CTA's logits are written
  unsigned long long best = 0;
  for (int r = rb0 * kTileR + tid; r < rb1 * kTileR; r += kNC) {
    const unsigned long long k = argmax_key(__ldcg(p.out + r), r);
    best = k > best ? k : best;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long k = __shfl_xor_sync(0xffffffffu, best, o);
    best = k > best ? k : best;
  }
  unsigned long long* red = reinterpret_cast<unsigned long long*>(W.part);
  if (lane == 0) red[warp] = best;
  named_barrier(1, kNC);
  if (tid == 0) {
    for (int w = 1; w < kConsumerWarps; ++w) best = red[w] > best ? red[w] : best;
    atomicMax(P.key, best);
    // release this CTA's maximum, acquire the others'
    unsigned long long t;
    asm volatile("atom.add.acq_rel.gpu.u64 %0, [%1], 1;" : "=l"(t) : "l"(P.key + 1) : "memory");
    if (t == (unsigned long long)(nb - 1)) {
      const unsigned long long k = atomicMax(P.key, 0ull);
      *P.token_out = (int)~(uint32_t)(k & 0xffffffffu);
      P.key[0] = 0;
      P.key[1] = 0;
    }
  }
}

const void* lm_head_kernel_ptr() { return (const void*)lm_head_argmax; }

// ---- two-phase kernels (the three-kernel layer) -------------------------------
// Shared memory: ring (nstages x slot_bytes) | mbarriers | one work area that
// the two phases use in turn.

size_t attn_oproj_smem_bytes(int hd, int G, int K_o, int max_rb_o, bool q4, int nstages,
                             int slot_bytes) {
  size_t work = AttnLayout{hd, G, kConsumerWarps}.total();
  const size_t g = GemvLayout{K_o, max_rb_o, q4}.total();
  if (g > work) work = g;
  return (size_t)nstages * slot_bytes + 16 * (size_t)nstages + work;
}

size_t ffn_smem_bytes(int K_gu, int max_rb_gu, int K_down, int max_rb_down, bool q4, int nstages,
                      int slot_bytes) {
  size_t work = GemvLayout{K_gu, max_rb_gu, q4}.total();
  const size_t g = GemvLayout{K_down, max_rb_down, q4}.total();
  if (g > work) work = g;
  return (size_t)nstages * slot_bytes + 16 * (size_t)nstages + work;
}

// Attention over the KV cache (the first att_grid CTAs; a flat split of every
// KV head's chunks, split heads merged by their last CTA through global
// memory), grid barrier, then o-proj + residual over every CTA.  The producer
// streams this CTA's K/V chunks and then its Wo slab without a break.
template <int HD, int G, bool Q4>
__global__ void __launch_bounds__(kThreads, 1) attn_oproj_fused(const AttnOprojParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Ring R{smem, reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * p.slot_bytes),
               reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * p.slot_bytes) + p.nstages,
               p.nstages, p.slot_bytes};
  uint8_t* work = smem + (size_t)p.nstages * p.slot_bytes + 16 * (size_t)p.nstages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  if (tid == 0) tl_mark_min(p.attn.tl, 0);
  // The step position, read before griddepcontrol.wait (see attn_decode): it
  // selects this step's barrier counter; the other one is cleared for the next.
  const int pos = *p.attn.pos;
  int* ctr = p.bar + (pos & 1);
  if (b == 0 && tid == 0) p.bar[(pos & 1) ^ 1] = 0;
  AttnSplit S = attn_split<HD>(pos, p.attn.nkv, b < p.att_grid ? b : 0, p.att_grid);
  if (b >= p.att_grid) S.u0 = S.u1 = S.U, S.nu = 0;
  const int rb0 = (int)split_begin(p.o.n_rb, nb, b), rb1 = (int)split_begin(p.o.n_rb, nb, b + 1);
  if (tid == 0) ring_init(R);
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      RingPos P{0, 0, 0};
      const uint64_t pol = policy_evict_first();
      attn_produce<HD>(p.attn, p.attn.kc, p.attn.vc, R, P, S, pol, [] { pdl_wait(); });
      gemv_produce(p.o, p.o.w, R, P, rb0, rb1, pol);
      l2_ahead(p.o.ahead, b);
    }
    return;
  }
  pdl_wait();  // q comes from the QKV kernel
  pdl_trigger();
  if (tid == 0) {
    tl_mark_min(p.attn.tl, 2);
    tl_mark_max(p.attn.tl, 3);
  }
  RingPos P{0, 0, 0};
  bool ok = attn_main<HD, G, false, kConsumerWarps>(p.attn, work, R, P, S, b, p.att_grid, tid);
  if (p.attn.tl) {
    named_barrier(1, kNC);
    if (tid == 0) {
      tl_mark_max(p.attn.tl, 1);
      tl_mark_min(p.attn.tl, 7);
    }
  }
  // every head is merged into o (by its last CTA) before any CTA reads o
  grid_sync(ctr, nb, p.attn.err, tid, 1, kNC, p.tl2);
  const GemvWork W(work, GemvLayout{p.o.geo.K, p.o.max_rb_local, Q4});
  gemv_pre<PRO_PLAIN>(p.o, nullptr, W, tid);
  GemvParams po = p.o;
  po.tl = p.tl2;
  ok &= gemv_main<PRO_PLAIN, EPI_RESID, Q4>(po, gemv_io(po), W, R, P, rb0, rb1, tid, b == 0);
  if (p.tl2) {
    named_barrier(1, kNC);
    if (tid == 0) {
      tl_mark_max(p.tl2, 1);
      tl_mark_min(p.tl2, 7);
    }
  }
  if (!ok && tid == 0) ring_drain(R, P, p.o.err);
}

// RMSNorm x weight, gate/up GEMV and SwiGLU (a to global memory), grid
// barrier, then the down GEMV + residual.  The producer streams this CTA's
// gate/up slab and then its down slab without a break.
template <bool Q4>
__global__ void __launch_bounds__(kThreads, 1) ffn_fused(const FfnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Ring R{smem, reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * p.slot_bytes),
               reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * p.slot_bytes) + p.nstages,
               p.nstages, p.slot_bytes};
  uint8_t* work = smem + (size_t)p.nstages * p.slot_bytes + 16 * (size_t)p.nstages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  if (tid == 0) tl_mark_min(p.gu.tl, 0);
  // The down phase of the last layer advances the step position; every CTA
  // reads it here, before the grid barrier that precedes that advance.
  const int pos = *p.gu.pos;
  int* ctr = p.bar + (pos & 1);
  if (b == 0 && tid == 0) p.bar[(pos & 1) ^ 1] = 0;
  const int ra0 = (int)split_begin(p.gu.n_rb, nb, b), ra1 = (int)split_begin(p.gu.n_rb, nb, b + 1);
  const int rd0 = (int)split_begin(p.down.n_rb, nb, b), rd1 = (int)split_begin(p.down.n_rb, nb, b + 1);
  if (tid == 0) ring_init(R);
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      RingPos P{0, 0, 0};
      const uint64_t pol = policy_evict_first();
      gemv_produce(p.gu, p.gu.w, R, P, ra0, ra1, pol);
      gemv_produce(p.down, p.down.w, R, P, rd0, rd1, pol);
      l2_ahead(p.down.ahead, b);
    }
    return;
  }
  const GemvWork W1(work, GemvLayout{p.gu.geo.K, p.gu.max_rb_local, Q4});
  gemv_pre<PRO_NORM>(p.gu, p.gu.norm_w, W1, tid);
  pdl_wait();  // h1 comes from the o-proj
  pdl_trigger();
  if (tid == 0) {
    tl_mark_min(p.gu.tl, 2);
    tl_mark_max(p.gu.tl, 3);
  }
  RingPos P{0, 0, 0};
  bool ok = gemv_main<PRO_NORM, EPI_SWIGLU, Q4>(p.gu, gemv_io(p.gu), W1, R, P, ra0, ra1, tid,
                                                 b == 0);
  if (p.gu.tl) {
    named_barrier(1, kNC);
    if (tid == 0) {
      tl_mark_max(p.gu.tl, 1);
      tl_mark_min(p.gu.tl, 7);
    }
  }
  // all of a is written before any CTA reads it
  grid_sync(ctr, nb, p.gu.err, tid, 1, kNC, p.tl2);
  const GemvWork W2(work, GemvLayout{p.down.geo.K, p.down.max_rb_local, Q4});
  gemv_pre<PRO_PLAIN>(p.down, nullptr, W2, tid);
  GemvParams pd = p.down;
  pd.tl = p.tl2;
  ok &= gemv_main<PRO_PLAIN, EPI_RESID, Q4>(pd, gemv_io(pd), W2, R, P, rd0, rd1, tid, b == 0);
  if (p.tl2) {
    named_barrier(1, kNC);
    if (tid == 0) {
      tl_mark_max(p.tl2, 1);
      tl_mark_min(p.tl2, 7);
    }
  }
  if (!ok && tid == 0) ring_drain(R, P, p.gu.err);
}

// ---- attention + o-projection by KV-head group (one cluster launch) -------------
size_t attn_headproj_smem_bytes(int hd, int G, bool q4, int nstages, int quads, int nkv) {
  const HeadProjLayout L{hd, G, quads, (nkv + 15) / 16, q4};
  return (size_t)nstages * kAttnStageBytes + 16 * (size_t)nstages + L.total();
}

template <int HD, int G, bool Q4>
__global__ void __launch_bounds__(kThreads, 1) attn_headproj(const AttnHeadProjParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Ring R{smem, reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * kAttnStageBytes),
               reinterpret_cast<uint64_t*>(smem + (size_t)p.nstages * kAttnStageBytes) + p.nstages,
               p.nstages, kAttnStageBytes};
  uint8_t* work = smem + (size_t)p.nstages * kAttnStageBytes + 16 * (size_t)p.nstages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  const int C = p.attn.cluster, r = (int)cluster_rank(), gh = b / C, nkv = p.attn.nkv;
  constexpr int Kg = G * HD;
  const int quads_max = (p.n_rb + C - 1) / C;
  const HeadProjLayout L{HD, G, quads_max, (nkv + 15) / 16, Q4};
  float* og = reinterpret_cast<float*>(work + L.og_off());
  uint64_t* bars = reinterpret_cast<uint64_t*>(work + L.bar_off());
  int* last_flag = reinterpret_cast<int*>(bars + 3);
  if (tid == 0) tl_mark_min(p.attn.tl, 0);
  const int pos = *p.attn.pos;  // see attn_decode
  const AttnSplit S = attn_split_cluster<HD>(pos, nkv, b, C);
  // this CTA's rows of the group's projection (the same split in every cluster)
  const int rb0 = (int)split_begin(p.n_rb, C, r), rb1 = (int)split_begin(p.n_rb, C, r + 1);
  if (tid == 0) {
    ring_init(R);
    for (int i = 0; i < 3; ++i) mbar_init(&bars[i], (uint32_t)C);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's exchange barriers exist before any remote arrival

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      RingPos P{0, 0, 0};
      const uint64_t pol = policy_evict_first();
      attn_produce<HD>(p.attn, p.attn.kc, p.attn.vc, R, P, S, pol, [] { pdl_wait(); });
      rows_produce(p.wo + (int64_t)gh * p.group_bytes, p.geo, rb0, rb1, R, P, pol, p.attn.err);
      l2_ahead(p.ahead, b);
    }
    return;
  }
  pdl_wait();  // q comes from the QKV kernel
  pdl_trigger();
  if (tid == 0) {
    tl_mark_min(p.attn.tl, 2);
    tl_mark_max(p.attn.tl, 3);
  }
  RingPos P{0, 0, 0};
  const ClusterXchg xg{og, bars};
  bool ok = attn_main<HD, G, true, kConsumerWarps, true>(p.attn, work, R, P, S, b, nb, tid, &xg);
  if (tid == 0) {
    tl_mark_max(p.attn.tl, 1);
    tl_mark_min(p.attn.tl, 7);
    tl_mark_min(p.tl2, 0);
    tl_mark_min(p.tl2, 2);
    tl_mark_max(p.tl2, 3);
  }
  // o_g is complete in this CTA: its int8 codes (q4), then rows [rb0, rb1) of
  // Wo_g o_g into the group's partial vector
  uint8_t* qx = work + L.qx_off();
  float* dx = reinterpret_cast<float*>(work + L.dx_off());
  int* sx = reinterpret_cast<int*>(work + L.sx_off());
  if (Q4) {
    quantize_blocks<false>(og, Kg, qx, dx, sx, (r == 0 && p.qtap) ? p.qtap + (size_t)gh * Kg : nullptr,
                    (r == 0 && p.qstap) ? p.qstap + (size_t)gh * (Kg / 32) : nullptr, tid, kNC,
                    1.0f);
    named_barrier(1, kNC);
  }
  float* part = p.part + (size_t)gh * p.n_rb * kTileR;
  ok &= rows_main<Q4>(p.geo, og, qx, dx, sx, R, P, rb0, rb1, tid, p.attn.err,
                      p.dots ? p.dots + (size_t)gh * (Kg / 32) : nullptr, nkv * (Kg / 32),
                      [&](int row, float v) { part[row] = v; });
  if (tid == 0) tl_mark_max(p.tl2, 6);
  // the CTA of rank r that finishes last over the groups adds up their rows
  named_barrier(1, kNC);
  if (tid == 0) {
    const int last = atomic_add_acq_rel(&p.cnt[r], 1) == nkv - 1;
    if (last) p.cnt[r] = 0;  // every group has arrived: ready for the next launch
    *last_flag = last;
  }
  named_barrier(1, kNC);
  if (*last_flag)
    headproj_sum(p.part, nkv, p.n_rb * kTileR, p.resid, p.out, p.tap, rb0 * kTileR, rb1 * kTileR,
                 reinterpret_cast<float4*>(work + L.red_off()), tid, kNC);
  // the other CTAs of the cluster have read this CTA's attention record
  if (!mbar_wait_cluster(&bars[2], 0, p.attn.err)) {
    raise_error(p.attn.err, ERR_CLUSTER_WAIT);
    ok = false;
  }
  if (tid == 0) {
    tl_mark_max(p.tl2, 1);
    tl_mark_min(p.tl2, 7);
  }
  if (!ok && tid == 0) ring_drain(R, P, p.attn.err);
}

const void* attn_headproj_kernel_ptr(int hd, int G, bool q4) {
#define TLD_HP(H_, G_)                                                    \
  if (hd == H_ && G == G_)                                                \
    return q4 ? (const void*)attn_headproj<H_, G_, true>                  \
              : (const void*)attn_headproj<H_, G_, false>;
  TLD_HP(64, 1) TLD_HP(64, 2) TLD_HP(64, 4) TLD_HP(64, 8)
  TLD_HP(128, 1) TLD_HP(128, 2) TLD_HP(128, 4) TLD_HP(128, 8)
#undef TLD_HP
  return nullptr;
}

const void* attn_oproj_kernel_ptr(int hd, int G, bool q4) {
#define TLD_AO(H_, G_)                                                    \
  if (hd == H_ && G == G_)                                                \
    return q4 ? (const void*)attn_oproj_fused<H_, G_, true>               \
              : (const void*)attn_oproj_fused<H_, G_, false>;
  TLD_AO(64, 1) TLD_AO(64, 2) TLD_AO(64, 4) TLD_AO(64, 8)
  TLD_AO(128, 1) TLD_AO(128, 2) TLD_AO(128, 4) TLD_AO(128, 8)
#undef TLD_AO
  return nullptr;
}

const void* ffn_kernel_ptr(bool q4) {
  return q4 ? (const void*)ffn_fused<true> : (const void*)ffn_fused<false>;
}

// ---- launch plumbing -----------------------------------------------------------

const void* gemv_kernel_ptr(int pro, int epi, bool q4) {
#define TLD_GEMV(P_, E_)                                                        \
  if (pro == P_ && epi == E_)                                                  \
    return q4 ? (const void*)gemv_fused<P_, E_, true> : (const void*)gemv_fused<P_, E_, false>;
  TLD_GEMV(PRO_NORM, EPI_QKV) TLD_GEMV(PRO_PLAIN, EPI_RESID) TLD_GEMV(PRO_NORM, EPI_SWIGLU)
#undef TLD_GEMV
  return nullptr;
}

const void* attn_kernel_ptr(int hd, int G, bool cluster) {
#define TLD_ATTN(H_, G_)                                                                       \
  if (hd == H_ && G == G_)                                                                    \
    return cluster ? (const void*)attn_decode<H_, G_, true, attn_warps(H_, G_, true)>     \
                   : (const void*)attn_decode<H_, G_, false, kAttnWarps>;
  TLD_ATTN(64, 1) TLD_ATTN(64, 2) TLD_ATTN(64, 4) TLD_ATTN(64, 8)
  TLD_ATTN(128, 1) TLD_ATTN(128, 2) TLD_ATTN(128, 4) TLD_ATTN(128, 8)
#undef TLD_ATTN
  return nullptr;
}

cudaError_t set_smem_limits() {
  const int max_smem = 227 * 1024;
  const void* ks[] = {gemv_kernel_ptr(PRO_NORM, EPI_QKV, false),
                      gemv_kernel_ptr(PRO_PLAIN, EPI_RESID, false),
                      gemv_kernel_ptr(PRO_NORM, EPI_SWIGLU, false),
                      gemv_kernel_ptr(PRO_NORM, EPI_QKV, true),
                      gemv_kernel_ptr(PRO_PLAIN, EPI_RESID, true),
                      gemv_kernel_ptr(PRO_NORM, EPI_SWIGLU, true)};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
  }
  {
    cudaError_t e = cudaFuncSetAttribute(lm_head_kernel_ptr(),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
  }
  for (bool q4 : {false, true}) {
    cudaError_t e = cudaFuncSetAttribute(ffn_kernel_ptr(q4),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
    for (int hd : {64, 128})
      for (int G : {1, 2, 4, 8}) {
        e = cudaFuncSetAttribute(attn_oproj_kernel_ptr(hd, G, q4),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (e != cudaSuccess) return e;
      }
  }
  for (int hd : {64, 128})
    for (int G : {1, 2, 4, 8})
      for (bool cl : {false, true}) {
        const void* k = attn_kernel_ptr(hd, G, cl);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (e == cudaSuccess && cl)
          e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
      }
  for (int hd : {64, 128})
    for (int G : {1, 2, 4, 8})
      for (bool q4 : {false, true}) {
        const void* k = attn_headproj_kernel_ptr(hd, G, q4);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

static cudaError_t launch_pdl(const void* fn, void** args, int grid, size_t smem, cudaStream_t s,
                              bool pdl, int cluster = 0, int threads = kThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_gemv(int pro, int epi, bool q4, const GemvParams& p, int grid, size_t smem,
                        cudaStream_t s, bool pdl) {
  const void* fn = gemv_kernel_ptr(pro, epi, q4);
  if (!fn) return cudaErrorInvalidValue;
  GemvParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(fn, args, grid, smem, s, pdl);
}

cudaError_t launch_attn(int hd, int G, const AttnParams& p, int grid, size_t smem,
                        cudaStream_t s, bool pdl) {
  const void* fn = attn_kernel_ptr(hd, G, p.cluster > 0);
  if (!fn) return cudaErrorInvalidValue;
  if (p.cluster > 0 && (p.cluster > kMaxCluster || grid != p.nkv * p.cluster))
    return cudaErrorInvalidValue;
  AttnParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(fn, args, grid, smem, s, pdl, p.cluster,
                    (attn_consumer_warps(hd, G, p.cluster > 0) + 1) * 32);
}

cudaError_t launch_lm_head(const LmHeadParams& p, int grid, size_t smem, cudaStream_t s, bool pdl) {
  LmHeadParams copy = p;
  void* args[] = {&copy};
  return launch_pdl((const void*)lm_head_argmax, args, grid, smem, s, pdl);
}

cudaError_t launch_attn_oproj(int hd, int G, bool q4, const AttnOprojParams& p, int grid,
                              size_t smem, cudaStream_t s, bool pdl) {
  const void* fn = attn_oproj_kernel_ptr(hd, G, q4);
  if (!fn || p.att_grid < 1 || p.att_grid > grid) return cudaErrorInvalidValue;
  AttnOprojParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(fn, args, grid, smem, s, pdl);
}

cudaError_t launch_attn_headproj(int hd, int G, bool q4, const AttnHeadProjParams& p, int grid,
                                 size_t smem, cudaStream_t s, bool pdl) {
  const void* fn = attn_headproj_kernel_ptr(hd, G, q4);
  if (!fn || p.attn.cluster < 1 || p.attn.cluster > kMaxCluster || grid != p.attn.nkv * p.attn.cluster)
    return cudaErrorInvalidValue;
  AttnHeadProjParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(fn, args, grid, smem, s, pdl, p.attn.cluster);
}

cudaError_t launch_ffn(bool q4, const FfnParams& p, int grid, size_t smem, cudaStream_t s,
                       bool pdl) {
  FfnParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(ffn_kernel_ptr(q4), args, grid, smem, s, pdl);
}

// ---- load-time repack ------------------------------------------------------------
__global__ void repack_bf16_kernel(const uint16_t* __restrict__ src, int rows, int K,
                                   uint16_t* __restrict__ dst, int dst_row0, int kind, int hd) {
  for (int s = blockIdx.x; s < rows; s += gridDim.x) {
    int64_t r;
    if (kind == 1) {
      const int head = s / hd, j = s % hd, half = hd / 2;
      const int local = head * hd + (j < half ? 2 * j : 2 * (j - half) + 1);
      r = dst_row0 + local;
    } else if (kind == 2) {
      r = dst_row0 + 2 * (int64_t)s;
    } else {
      r = dst_row0 + s;
    }
    const uint16_t* in = src + (size_t)s * K;
    for (int k = threadIdx.x; k < K; k += blockDim.x) dst[tiled_elem_offset(r, k, K)] = in[k];
  }
}

cudaError_t launch_repack_bf16(const uint16_t* src, int rows, int K, uint8_t* dst_tiled,
                               int dst_row0, int kind, int hd, cudaStream_t s) {
  const int grid = rows < 4096 ? rows : 4096;
  repack_bf16_kernel<<<grid, 256, 0, s>>>(src, rows, K, reinterpret_cast<uint16_t*>(dst_tiled),
                                          dst_row0, kind, hd);
  return cudaGetLastError();
}

__device__ __forceinline__ int64_t repack_row(int s, int dst_row0, int kind, int hd) {
  if (kind == 1) {
    const int head = s / hd, j = s % hd, half = hd / 2;
    return dst_row0 + head * hd + (j < half ? 2 * j : 2 * (j - half) + 1);
  }
  if (kind == 2) return dst_row0 + 2 * (int64_t)s;
  return dst_row0 + s;
}

__global__ void repack_q4_kernel(const uint8_t* __restrict__ nib, const uint16_t* __restrict__ sc,
                                 int rows, int K, uint8_t* __restrict__ dst, int dst_row0, int kind,
                                 int hd) {
  for (int s = blockIdx.x; s < rows; s += gridDim.x) {
    const int64_t r = repack_row(s, dst_row0, kind, hd);
    if (nib) {
      const uint8_t* in = nib + (size_t)s * (K / 2);
      for (int c2 = threadIdx.x; c2 < K / 2; c2 += blockDim.x) dst[q4_nibble_byte(r, c2, K)] = in[c2];
    }
    if (sc) {
      const uint16_t* in = sc + (size_t)s * (K / 32);
      for (int bb = threadIdx.x; bb < K / 32; bb += blockDim.x)
        *reinterpret_cast<uint16_t*>(dst + q4_scale_byte(r, bb, K)) = in[bb];
    }
  }
}

// Wo split by KV-head group: columns [g*Kg, (g+1)*Kg) of each row go to group
// g's tiled matrix of K = Kg at dst + g * group_bytes.
__global__ void repack_groups_kernel(const uint8_t* __restrict__ src, int mode, int rows, int K,
                                     int Kg, uint8_t* __restrict__ dst, int64_t group_bytes) {
  for (int s = blockIdx.x; s < rows; s += gridDim.x) {
    if (mode == 0) {  // bf16 elements
      const uint16_t* in = reinterpret_cast<const uint16_t*>(src) + (size_t)s * K;
      for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const int g = k / Kg, kk = k - g * Kg;
        reinterpret_cast<uint16_t*>(dst + g * group_bytes)[tiled_elem_offset(s, kk, Kg)] = in[k];
      }
    } else if (mode == 1) {  // q4 nibble pairs
      const uint8_t* in = src + (size_t)s * (K / 2);
      for (int c2 = threadIdx.x; c2 < K / 2; c2 += blockDim.x) {
        const int g = (2 * c2) / Kg, cc = c2 - g * (Kg / 2);
        dst[g * group_bytes + q4_nibble_byte(s, cc, Kg)] = in[c2];
      }
    } else {  // q4 block scales
      const uint16_t* in = reinterpret_cast<const uint16_t*>(src) + (size_t)s * (K / 32);
      for (int bb = threadIdx.x; bb < K / 32; bb += blockDim.x) {
        const int g = (32 * bb) / Kg, bg = bb - g * (Kg / 32);
        *reinterpret_cast<uint16_t*>(dst + g * group_bytes + q4_scale_byte(s, bg, Kg)) = in[bb];
      }
    }
  }
}

cudaError_t launch_repack_groups(const void* src, bool q4_scales, bool q4, int rows, int K, int Kg,
                                 uint8_t* dst, int64_t group_bytes, cudaStream_t s) {
  const int grid = rows < 4096 ? rows : 4096;
  repack_groups_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint8_t*>(src),
                                            !q4 ? 0 : q4_scales ? 2 : 1, rows, K, Kg, dst, group_bytes);
  return cudaGetLastError();
}

cudaError_t launch_repack_q4(const uint8_t* nibbles, const uint16_t* scales, int rows, int K,
                             uint8_t* dst_tiled, int dst_row0, int kind, int hd, cudaStream_t s) {
  const int grid = rows < 4096 ? rows : 4096;
  repack_q4_kernel<<<grid, 256, 0, s>>>(nibbles, scales, rows, K, dst_tiled, dst_row0, kind, hd);
  return cudaGetLastError();
}

}  // namespace tld
