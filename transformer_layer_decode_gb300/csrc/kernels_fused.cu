// Fused decode-layer kernels for sm_103a.
//
// Five kernels per layer (the fusions of "RDNA4 Decode Kernel Fusion:
// Pipeline Barriers, Not Launches, Are the Win", FAQ and section "Fusion
// removes the barrier by removing the write"):
//   K1 gemv<PRO_NORM,  EPI_QKV>    RMSNorm*w prologue, [Wq;Wk;Wv] GEMV, RoPE on
//                                  q and k and the k/v append in the epilogue
//   K2 attn_decode                 GQA split-KV attention + last-CTA combine
//   K3 gemv<PRO_PLAIN, EPI_RESID>  Wo GEMV + residual add
//   K4 gemv<PRO_NORM,  EPI_SWIGLU> RMSNorm*w prologue, interleaved gate/up GEMV,
//                                  silu(g)*u in the epilogue (g, u never stored)
//   K5 gemv<PRO_PLAIN, EPI_RESID>  Wd GEMV + residual add
//
// Batch-1 projections are matrix-vector products: one flop per weight byte, so
// they are bound by HBM, not by the tensor cores.  Each GEMV CTA owns one
// contiguous slab of the tiled weight matrix (a balanced split of its tiles
// over the grid) and streams it through a ring of 16 KB shared-memory stages
// filled by 1-D bulk copies (TMA) issued by one producer thread; eight
// consumer warps each take one 4-row x 256-column tile per stage, read the
// input vector from shared memory and accumulate in fp32.  A row block cut by
// the split is finished by the last CTA to arrive (atomic ticket, partials
// summed in CTA order, so results are deterministic).  Weights do not depend
// on the previous kernel, so the producer starts streaming before
// griddepcontrol.wait; only the input vector waits for the previous kernel.
#include "common.cuh"
#include "kernels.h"

namespace tld {

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// ---- shared memory layout of the GEMV kernel -------------------------------
struct GemvSmem {
  int K, nstages, max_rb_local;
  __host__ __device__ size_t stages_off() const { return 0; }
  __host__ __device__ size_t bars_off() const { return (size_t)nstages * kStageBytes; }
  __host__ __device__ size_t xs_off() const { return bars_off() + 2 * 8 * (size_t)nstages; }
  __host__ __device__ size_t part_off() const { return xs_off() + 4 * (size_t)((K + 3) & ~3); }
  __host__ __device__ size_t red_off() const {
    return part_off() + 4 * (size_t)max_rb_local * kConsumerWarps * kTileR;
  }
  __host__ __device__ size_t total() const { return red_off() + 4 * 32 + 16; }  // red[0..8]: warp sums + abort mark
};

size_t gemv_smem_bytes(int K, int nstages, int max_rb_local) {
  return GemvSmem{K, nstages, max_rb_local}.total();
}

// Epilogue of one finished row block (4 tiled rows, values v).
template <int EPI>
__device__ __forceinline__ void gemv_epilogue(const GemvParams& p, int rb, const float v[4]) {
  const int R0 = rb * kTileR;
  if (EPI == EPI_QKV) {
    const int hd = p.hd, half = hd / 2;
    const int qrows = p.nq * hd, krows = p.nkv * hd;
    const int pos = *p.pos;
    if (R0 < qrows + krows) {
      const bool is_q = R0 < qrows;
      const int local = is_q ? R0 : R0 - qrows;
      const int head = local / hd, i0 = (local % hd) / 2;  // two rope pairs: i0, i0+1
      const float2* cs = p.rope + (size_t)pos * half;
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        const int i = i0 + pr;
        const float a = v[2 * pr], b = v[2 * pr + 1];
        const float2 c = cs[i];
        const float ra = a * c.x - b * c.y;
        const float rb2 = a * c.y + b * c.x;
        if (is_q) {
          p.q_out[head * hd + i] = ra;
          p.q_out[head * hd + i + half] = rb2;
        } else {
          uint16_t* row = p.kc + ((size_t)head * p.max_ctx + pos) * hd;
          row[i] = f32_to_bf16_bits(ra);
          row[i + half] = f32_to_bf16_bits(rb2);
        }
      }
    } else {
      const int local = R0 - qrows - krows;
      const int head = local / hd, j = local % hd;
      uint16_t* row = p.vc + ((size_t)head * p.max_ctx + pos) * hd;
#pragma unroll
      for (int r = 0; r < 4; ++r) row[j + r] = f32_to_bf16_bits(v[r]);
    }
  } else if (EPI == EPI_RESID) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float y = p.resid[R0 + r] + v[r];
      p.out[R0 + r] = y;
      if (p.tap) p.tap[R0 + r] = y;
    }
  } else {  // EPI_SWIGLU: tiled rows (g_j, u_j, g_j+1, u_j+1)
    const int j = R0 / 2;
    p.a_out[j] = silu_f(v[0]) * v[1];
    p.a_out[j + 1] = silu_f(v[2]) * v[3];
  }
}

// Reduce 4 per-lane row accumulators over the warp; lane 8r ends with row r.
__device__ __forceinline__ float warp_reduce4(const float a[4], int lane) {
  const bool hi = lane & 16;
  float keep0 = hi ? a[2] : a[0], keep1 = hi ? a[3] : a[1];
  const float send0 = hi ? a[0] : a[2], send1 = hi ? a[1] : a[3];
  keep0 += __shfl_xor_sync(0xffffffffu, send0, 16);
  keep1 += __shfl_xor_sync(0xffffffffu, send1, 16);
  const bool b3 = lane & 8;
  float k = b3 ? keep1 : keep0;
  const float snd = b3 ? keep0 : keep1;
  k += __shfl_xor_sync(0xffffffffu, snd, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

template <int PRO, int EPI>
__global__ void __launch_bounds__(kThreads, 2) gemv_fused(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GemvSmem L{p.K, p.nstages, p.max_rb_local};
  uint8_t* stages = smem + L.stages_off();
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars_off());
  uint64_t* empty = full + p.nstages;
  float* xs = reinterpret_cast<float*>(smem + L.xs_off());
  float* part_s = reinterpret_cast<float*>(smem + L.part_off());
  float* red = reinterpret_cast<float*>(smem + L.red_off());

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  const int64_t t0 = split_begin(p.ntiles, nb, b), t1 = split_begin(p.ntiles, nb, b + 1);
  const int nloc = (int)(t1 - t0);
  const int nst = (nloc + kStageTiles - 1) / kStageTiles;

  if (tid == 0) {
    for (int s = 0; s < p.nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---- producer: stream this CTA's slab (weights only: no wait needed) ----
    if (lane == 0) {
      for (int s = 0; s < nst; ++s) {
        const int slot = s % p.nstages;
        if (s >= p.nstages && !mbar_wait(&empty[slot], ((s / p.nstages) - 1) & 1)) {
          raise_error(p.err, ERR_EMPTY_WAIT);
          break;
        }
        const int64_t ta = t0 + (int64_t)s * kStageTiles;
        const int64_t tb = min(ta + kStageTiles, t1);
        const int64_t oa = tile_byte_offset(ta, p.ktiles, p.K);
        const uint32_t bytes = (uint32_t)(tile_byte_offset(tb, p.ktiles, p.K) - oa);
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(stages + (size_t)slot * kStageBytes, p.w + oa, bytes, &full[slot]);
      }
    }
    return;
  }

  // ---- consumers -------------------------------------------------------------
  pdl_wait();  // the input vector comes from the previous kernel
  // Let the next kernel launch (and prefetch its weights) now.  Triggering only
  // after this CTA's own wait keeps at most two kernels in flight and means that
  // everything before the previous kernel is complete when the next one starts.
  pdl_trigger();
  constexpr int NC = kConsumerWarps * 32;
  if (tid == 0) red[kConsumerWarps] = 0.f;
  if (PRO == PRO_NORM) {
    float ss = 0.f;
    const float4* x4 = reinterpret_cast<const float4*>(p.x);
    for (int k4 = tid; k4 < p.K / 4; k4 += NC) {
      const float4 v = x4[k4];
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    named_barrier(1, NC);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += red[w];
    const float r = 1.0f / sqrtf(tot / (float)p.K + p.eps);
    const uint2* w4 = reinterpret_cast<const uint2*>(p.norm_w);
    for (int k4 = tid; k4 < p.K / 4; k4 += NC) {
      const float4 v = x4[k4];
      const uint2 wb = w4[k4];
      float4 o;
      o.x = v.x * r * bf16lo(wb.x);
      o.y = v.y * r * bf16hi(wb.x);
      o.z = v.z * r * bf16lo(wb.y);
      o.w = v.w * r * bf16hi(wb.y);
      reinterpret_cast<float4*>(xs)[k4] = o;
    }
  } else {
    const float4* x4 = reinterpret_cast<const float4*>(p.x);
    for (int k4 = tid; k4 < p.K / 4; k4 += NC) reinterpret_cast<float4*>(xs)[k4] = x4[k4];
  }
  if (p.x_copy && b == 0) {
    for (int k = tid; k < p.K; k += NC) p.x_copy[k] = p.x[k];
  }
  if (p.pos_advance && b == 0 && tid == 0) atomicAdd(p.pos_advance, 1);
  for (int i = tid; i < p.max_rb_local * kConsumerWarps * kTileR; i += NC) part_s[i] = 0.f;
  named_barrier(1, NC);

  const int rb_first = nloc > 0 ? (int)(t0 / p.ktiles) : 0;
  int cur_rb = -1;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool ok = true;
  for (int s = 0; s < nst; ++s) {
    const int slot = s % p.nstages;
    // After a timed-out wait the warp stops waiting but keeps the same control
    // flow, so that every named barrier below is still reached by all warps.
    if (ok && !mbar_wait(&full[slot], (s / p.nstages) & 1)) {
      raise_error(p.err, ERR_FULL_WAIT);
      ok = false;
    }
    const int li = s * kStageTiles + warp;
    if (li < nloc) {
      const int64_t t = t0 + li;
      const int rb = (int)(t / p.ktiles), kt = (int)(t - (int64_t)rb * p.ktiles);
      if (rb != cur_rb) {
        if (cur_rb >= 0) {
          const float v = warp_reduce4(acc, lane);
          if ((lane & 7) == 0)
            part_s[((cur_rb - rb_first) * kConsumerWarps + warp) * kTileR + (lane >> 3)] = v;
        }
        cur_rb = rb;
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      }
      const int kw = (kt == p.ktiles - 1) ? p.kw_last : kTileK;
      const int64_t sa = t0 + (int64_t)s * kStageTiles;
      const uint8_t* tp = stages + (size_t)slot * kStageBytes +
                          (tile_byte_offset(t, p.ktiles, p.K) - tile_byte_offset(sa, p.ktiles, p.K));
      const int c = lane * 8;
      if (c < kw) {
        const float4 xa = *reinterpret_cast<const float4*>(xs + kt * kTileK + c);
        const float4 xb = *reinterpret_cast<const float4*>(xs + kt * kTileK + c + 4);
#pragma unroll
        for (int r = 0; r < kTileR; ++r) {
          const uint4 wv = *reinterpret_cast<const uint4*>(tp + ((size_t)r * kw + c) * 2);
          float a = acc[r];
          a = fmaf(bf16lo(wv.x), xa.x, a);
          a = fmaf(bf16hi(wv.x), xa.y, a);
          a = fmaf(bf16lo(wv.y), xa.z, a);
          a = fmaf(bf16hi(wv.y), xa.w, a);
          a = fmaf(bf16lo(wv.z), xb.x, a);
          a = fmaf(bf16hi(wv.z), xb.y, a);
          a = fmaf(bf16lo(wv.w), xb.z, a);
          a = fmaf(bf16hi(wv.w), xb.w, a);
          acc[r] = a;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  if (cur_rb >= 0) {
    const float v = warp_reduce4(acc, lane);
    if ((lane & 7) == 0)
      part_s[((cur_rb - rb_first) * kConsumerWarps + warp) * kTileR + (lane >> 3)] = v;
  }
  if (!ok && lane == 0) red[kConsumerWarps] = 1.f;  // abort mark
  named_barrier(1, NC);
  if (red[kConsumerWarps] != 0.f) {
    // Drain: wait (bounded) for the last copy into every slot, then leave.
    if (tid == 0)
      for (int s = 0; s < nst && s < p.nstages; ++s) {
        const int last = s + ((nst - 1 - s) / p.nstages) * p.nstages;
        if (!mbar_wait(&full[s], (last / p.nstages) & 1)) raise_error(p.err, ERR_DRAIN);
      }
    return;
  }
  if (nloc == 0) return;

  // ---- finish row blocks ------------------------------------------------------
  const int rb_last = (int)((t1 - 1) / p.ktiles);
  for (int j = tid; j <= rb_last - rb_first; j += NC) {
    const int rb = rb_first + j;
    float v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float s = 0.f;
      for (int w = 0; w < kConsumerWarps; ++w) s += part_s[(j * kConsumerWarps + w) * kTileR + r];
      v[r] = s;
    }
    const int64_t rb_t0 = (int64_t)rb * p.ktiles, rb_t1 = rb_t0 + p.ktiles;
    if (rb_t0 >= t0 && rb_t1 <= t1) {
      gemv_epilogue<EPI>(p, rb, v);
      continue;
    }
    // split row block: publish, take a ticket, the last arrival finishes it
    const int side = (j == 0) ? 0 : 1;
    float* mine = p.part + ((size_t)b * 2 + side) * kTileR;
#pragma unroll
    for (int r = 0; r < 4; ++r) mine[r] = v[r];
    __threadfence();
    const int c_lo = split_owner(p.ntiles, nb, rb_t0), c_hi = split_owner(p.ntiles, nb, rb_t1 - 1);
    int expected = 0;
    for (int c = c_lo; c <= c_hi; ++c)
      expected += split_begin(p.ntiles, nb, c + 1) > split_begin(p.ntiles, nb, c);
    const int prev = atomicAdd(&p.counters[rb], 1);
    if (prev != expected - 1) continue;
    __threadfence();
    float tot[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = c_lo; c <= c_hi; ++c) {
      const int64_t cs = split_begin(p.ntiles, nb, c), ce = split_begin(p.ntiles, nb, c + 1);
      if (ce <= cs) continue;
      const int sd = (cs / p.ktiles == rb) ? 0 : 1;
      const float* q = p.part + ((size_t)c * 2 + sd) * kTileR;
#pragma unroll
      for (int r = 0; r < 4; ++r) tot[r] += __ldcg(q + r);
    }
    gemv_epilogue<EPI>(p, rb, tot);
    p.counters[rb] = 0;
  }
}

// ---- attention ---------------------------------------------------------------
// One unit = one chunk of CH cached positions of one KV head (K and V rows,
// 8 KB each).  The grid splits the units of all KV heads evenly; every CTA
// serves all G query heads of the KV heads it touches, so each K/V byte is
// read once.  Within a CTA the 8 consumer warps take interleaved positions of
// each chunk and keep a running (max, sum, acc) per query head; warps are
// merged at the end of each head segment, and a head cut between CTAs is
// merged by the last CTA to arrive, in CTA order.

struct AttnSmem {
  int hd, G, nstages;
  __host__ __device__ size_t bars_off() const { return (size_t)nstages * 16384; }
  __host__ __device__ size_t ws_off() const { return bars_off() + 16 * (size_t)nstages; }
  __host__ __device__ size_t seg_off() const {
    return ws_off() + 4 * (size_t)kConsumerWarps * G * (hd + 2);
  }
  __host__ __device__ size_t flag_off() const { return seg_off() + 4 * (size_t)G * (hd + 2); }
  __host__ __device__ size_t total() const { return flag_off() + 16; }
};

size_t attn_smem_bytes(int hd, int G, int nstages) { return AttnSmem{hd, G, nstages}.total(); }

template <int HD, int G>
__global__ void __launch_bounds__(kThreads, 2) attn_decode(const AttnParams p) {
  constexpr int CH = 8192 / (HD * 2);  // positions per chunk (8 KB of K)
  constexpr int PW = CH / kConsumerWarps;  // positions per warp per chunk
  constexpr int DL = HD / 32;          // dims per lane
  constexpr int NC = kConsumerWarps * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const AttnSmem L{HD, G, p.nstages};
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars_off());
  uint64_t* empty = full + p.nstages;
  float* ws = reinterpret_cast<float*>(smem + L.ws_off());    // [warp][G][HD+2]
  float* seg = reinterpret_cast<float*>(smem + L.seg_off());  // [G][HD+2]
  int* flag = reinterpret_cast<int*>(smem + L.flag_off());

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  // The step position is read before griddepcontrol.wait: it was last written by
  // the previous step's final kernel, and this kernel can only launch after the
  // preceding kernel's CTAs have all passed their own wait, i.e. after that
  // final kernel completed.
  const int pos = *p.pos;
  const int n = pos + 1;
  const int cph = (n + CH - 1) / CH;
  const int64_t U = (int64_t)p.nkv * cph;
  const int64_t u0 = split_begin(U, nb, b), u1 = split_begin(U, nb, b + 1);
  const int nu = (int)(u1 - u0);

  if (tid == 0) {
    for (int s = 0; s < p.nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      bool waited = false;
      for (int s = 0; s < nu; ++s) {
        const int slot = s % p.nstages;
        if (s >= p.nstages && !mbar_wait(&empty[slot], ((s / p.nstages) - 1) & 1)) {
          raise_error(p.err, ERR_EMPTY_WAIT);
          break;
        }
        const int64_t u = u0 + s;
        const int g = (int)(u / cph), c = (int)(u - (int64_t)g * cph);
        const int rows = min(CH, n - c * CH);
        if (c == cph - 1 && !waited) {  // this chunk holds the row appended by K1
          pdl_wait();
          waited = true;
        }
        const size_t off = ((size_t)g * p.max_ctx + (size_t)c * CH) * HD;
        const uint32_t bytes = (uint32_t)rows * HD * 2;
        mbar_arrive_expect_tx(&full[slot], 2 * bytes);
        uint8_t* dst = stages + (size_t)slot * 16384;
        bulk_g2s(dst, p.kc + off, bytes, &full[slot]);
        bulk_g2s(dst + 8192, p.vc + off, bytes, &full[slot]);
      }
    }
    return;
  }

  pdl_wait();  // q comes from K1
  pdl_trigger();
  float m[G], l[G], acc[G][DL];
  int cur_g = -1, seg_idx = 0;
  auto reset = [&]() {
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      m[gg] = -INFINITY;
      l[gg] = 0.f;
#pragma unroll
      for (int j = 0; j < DL; ++j) acc[gg][j] = 0.f;
    }
  };
  float qr[G][DL];
  // Ends the segment of KV head g: merge warps, then finish or publish.
  auto end_segment = [&](int g) {
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      float* w = ws + ((size_t)warp * G + gg) * (HD + 2);
#pragma unroll
      for (int j = 0; j < DL; ++j) w[lane * DL + j] = acc[gg][j];
      if (lane == 0) {
        w[HD] = m[gg];
        w[HD + 1] = l[gg];
      }
    }
    named_barrier(1, NC);
    for (int i = tid; i < G * HD; i += NC) {
      const int gg = i / HD, j = i % HD;
      float M = -INFINITY;
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, ws[(w * G + gg) * (HD + 2) + HD]);
      float A = 0.f, Ls = 0.f;
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* wr = ws + (w * G + gg) * (HD + 2);
        const float e = (wr[HD] == -INFINITY) ? 0.f : expf(wr[HD] - M);
        A += wr[j] * e;
        Ls += wr[HD + 1] * e;
      }
      seg[gg * (HD + 2) + j] = A;
      if (j == 0) {
        seg[gg * (HD + 2) + HD] = M;
        seg[gg * (HD + 2) + HD + 1] = Ls;
      }
    }
    named_barrier(1, NC);
    const int64_t h0 = (int64_t)g * cph, h1 = h0 + cph;
    if (h0 >= u0 && h1 <= u1) {  // whole head in this CTA
      for (int i = tid; i < G * HD; i += NC) {
        const int gg = i / HD, j = i % HD;
        p.o[(size_t)(g * G + gg) * HD + j] = seg[gg * (HD + 2) + j] / seg[gg * (HD + 2) + HD + 1];
      }
    } else {
      const int side = seg_idx == 0 ? 0 : 1;
      float* mine = p.part + ((size_t)b * 2 + side) * G * (HD + 2);
      for (int i = tid; i < G * (HD + 2); i += NC) mine[i] = seg[i];
      __threadfence();
      named_barrier(1, NC);
      if (tid == 0) {
        const int c_lo = split_owner(U, nb, h0), c_hi = split_owner(U, nb, h1 - 1);
        int expected = 0;
        for (int c = c_lo; c <= c_hi; ++c)
          expected += split_begin(U, nb, c + 1) > split_begin(U, nb, c);
        const int prev = atomicAdd(&p.counters[g], 1);
        *flag = (prev == expected - 1);
        if (*flag) __threadfence();
      }
      named_barrier(1, NC);
      if (*flag) {
        const int c_lo = split_owner(U, nb, h0), c_hi = split_owner(U, nb, h1 - 1);
        for (int i = tid; i < G * HD; i += NC) {
          const int gg = i / HD, j = i % HD;
          float M = -INFINITY;
          for (int c = c_lo; c <= c_hi; ++c) {
            const int64_t cs = split_begin(U, nb, c), ce = split_begin(U, nb, c + 1);
            if (ce <= cs) continue;
            const int sd = (cs >= h0) ? 0 : 1;
            M = fmaxf(M, __ldcg(p.part + (((size_t)c * 2 + sd) * G + gg) * (HD + 2) + HD));
          }
          float A = 0.f, Ls = 0.f;
          for (int c = c_lo; c <= c_hi; ++c) {
            const int64_t cs = split_begin(U, nb, c), ce = split_begin(U, nb, c + 1);
            if (ce <= cs) continue;
            const int sd = (cs >= h0) ? 0 : 1;
            const float* pr = p.part + (((size_t)c * 2 + sd) * G + gg) * (HD + 2);
            const float e = expf(__ldcg(pr + HD) - M);
            A += __ldcg(pr + j) * e;
            Ls += __ldcg(pr + HD + 1) * e;
          }
          p.o[(size_t)(g * G + gg) * HD + j] = A / Ls;
        }
        if (tid == 0) p.counters[g] = 0;
      }
    }
    named_barrier(1, NC);
    ++seg_idx;
  };

  reset();
  bool ok = true;
  for (int s = 0; s < nu; ++s) {
    const int slot = s % p.nstages;
    const int64_t u = u0 + s;
    const int g = (int)(u / cph), c = (int)(u - (int64_t)g * cph);
    if (g != cur_g) {
      if (cur_g >= 0) {
        end_segment(cur_g);
        reset();
      }
      cur_g = g;
#pragma unroll
      for (int gg = 0; gg < G; ++gg)
#pragma unroll
        for (int j = 0; j < DL; ++j) qr[gg][j] = p.q[(size_t)(g * G + gg) * HD + lane * DL + j] * p.scale;
    }
    if (ok && !mbar_wait(&full[slot], (s / p.nstages) & 1)) {
      raise_error(p.err, ERR_FULL_WAIT);
      ok = false;  // keep the control flow (segment barriers) uniform
    }
    const int rows = min(CH, n - c * CH);
    const uint8_t* kb = stages + (size_t)slot * 16384;
    const uint8_t* vb = kb + 8192;
    float sc[PW][G];
#pragma unroll
    for (int i = 0; i < PW; ++i) {
      const int t = warp + i * kConsumerWarps;
      float kv[DL];
      if (t < rows) {
        if (DL == 4) {
          const uint2 w2 = *reinterpret_cast<const uint2*>(kb + ((size_t)t * HD + lane * 4) * 2);
          kv[0] = bf16lo(w2.x); kv[1] = bf16hi(w2.x); kv[2] = bf16lo(w2.y); kv[3] = bf16hi(w2.y);
        } else {
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(kb + ((size_t)t * HD + lane * 2) * 2);
          kv[0] = bf16lo(w1); kv[1] = bf16hi(w1);
        }
      } else {
#pragma unroll
        for (int j = 0; j < DL; ++j) kv[j] = 0.f;
      }
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < DL; ++j) d = fmaf(qr[gg][j], kv[j], d);
        d = warp_sum(d);
        sc[i][gg] = (t < rows) ? d : -INFINITY;
      }
    }
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      float mx = m[gg];
#pragma unroll
      for (int i = 0; i < PW; ++i) mx = fmaxf(mx, sc[i][gg]);
      if (mx == -INFINITY) continue;  // this warp has no position in the chunk
      const float alpha = (m[gg] == -INFINITY) ? 0.f : expf(m[gg] - mx);
      float ls = l[gg] * alpha;
#pragma unroll
      for (int j = 0; j < DL; ++j) acc[gg][j] *= alpha;
#pragma unroll
      for (int i = 0; i < PW; ++i) {
        const int t = warp + i * kConsumerWarps;
        if (t >= rows) continue;
        const float pi = expf(sc[i][gg] - mx);
        ls += pi;
        float vv[DL];
        if (DL == 4) {
          const uint2 w2 = *reinterpret_cast<const uint2*>(vb + ((size_t)t * HD + lane * 4) * 2);
          vv[0] = bf16lo(w2.x); vv[1] = bf16hi(w2.x); vv[2] = bf16lo(w2.y); vv[3] = bf16hi(w2.y);
        } else {
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vb + ((size_t)t * HD + lane * 2) * 2);
          vv[0] = bf16lo(w1); vv[1] = bf16hi(w1);
        }
#pragma unroll
        for (int j = 0; j < DL; ++j) acc[gg][j] = fmaf(pi, vv[j], acc[gg][j]);
      }
      m[gg] = mx;
      l[gg] = ls;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  if (cur_g >= 0) end_segment(cur_g);
  if (!ok) {
    for (int s = 0; s < nu && s < p.nstages; ++s) {
      const int last = s + ((nu - 1 - s) / p.nstages) * p.nstages;
      if (!mbar_wait(&full[s], (last / p.nstages) & 1)) raise_error(p.err, ERR_DRAIN);
    }
  }
}

// ---- launch plumbing -----------------------------------------------------------

const void* gemv_kernel_ptr(int pro, int epi) {
  if (pro == PRO_NORM && epi == EPI_QKV) return (const void*)gemv_fused<PRO_NORM, EPI_QKV>;
  if (pro == PRO_PLAIN && epi == EPI_RESID) return (const void*)gemv_fused<PRO_PLAIN, EPI_RESID>;
  if (pro == PRO_NORM && epi == EPI_SWIGLU) return (const void*)gemv_fused<PRO_NORM, EPI_SWIGLU>;
  return nullptr;
}

const void* attn_kernel_ptr(int hd, int G) {
#define TLD_ATTN(H_, G_) \
  if (hd == H_ && G == G_) return (const void*)attn_decode<H_, G_>;
  TLD_ATTN(64, 1) TLD_ATTN(64, 2) TLD_ATTN(64, 4) TLD_ATTN(64, 8)
  TLD_ATTN(128, 1) TLD_ATTN(128, 2) TLD_ATTN(128, 4) TLD_ATTN(128, 8)
#undef TLD_ATTN
  return nullptr;
}

cudaError_t set_smem_limits() {
  const int max_smem = 227 * 1024;
  const void* ks[] = {gemv_kernel_ptr(PRO_NORM, EPI_QKV), gemv_kernel_ptr(PRO_PLAIN, EPI_RESID),
                      gemv_kernel_ptr(PRO_NORM, EPI_SWIGLU)};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
  }
  for (int hd : {64, 128})
    for (int G : {1, 2, 4, 8}) {
      cudaError_t e = cudaFuncSetAttribute(attn_kernel_ptr(hd, G),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

static cudaError_t launch_pdl(const void* fn, void** args, int grid, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_gemv(int pro, int epi, const GemvParams& p, int grid, size_t smem,
                        cudaStream_t s) {
  const void* fn = gemv_kernel_ptr(pro, epi);
  if (!fn) return cudaErrorInvalidValue;
  GemvParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(fn, args, grid, smem, s);
}

cudaError_t launch_attn(int hd, int G, const AttnParams& p, int grid, size_t smem,
                        cudaStream_t s) {
  const void* fn = attn_kernel_ptr(hd, G);
  if (!fn) return cudaErrorInvalidValue;
  AttnParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(fn, args, grid, smem, s);
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

}  // namespace tld
