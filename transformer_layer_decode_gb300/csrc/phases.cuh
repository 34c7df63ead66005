// Device-side phases of the decode layer, shared by the five-kernel plan
// (one phase per kernel launch) and the persistent per-token kernel (all
// phases of all layers in one launch, separated by grid barriers).
//
// Every phase streams its bytes (weights, or K/V rows) through one ring of
// shared-memory stages: a producer thread fills stages with 1-D bulk copies
// (TMA) that complete on the stage's "full" mbarrier; the consumer warps (eight;
// sixteen in some attention kernels) copy their part of a stage to registers,
// arrive on its "empty" mbarrier and compute.  A ring position counts stages since the ring was initialised, so
// one ring can carry the stages of many phases back to back.
#pragma once
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace tld {

constexpr int kNC = kConsumerWarps * 32;  // consumer threads

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// ---- the stage ring ----------------------------------------------------------
struct Ring {
  uint8_t* stages;
  uint64_t* full;
  uint64_t* empty;
  int n, slot_bytes;
  __device__ __forceinline__ uint8_t* slot(int s) const { return stages + (size_t)s * slot_bytes; }
};

struct RingPos {
  int slot, phase, count;  // count = stages passed since the ring was initialised
  __device__ __forceinline__ void next(int n) {
    ++count;
    if (++slot == n) {
      slot = 0;
      phase ^= 1;
    }
  }
};

__device__ __forceinline__ void ring_init(const Ring& R, int consumer_warps = kConsumerWarps) {
  for (int s = 0; s < R.n; ++s) {
    mbar_init(&R.full[s], 1);
    mbar_init(&R.empty[s], consumer_warps);
  }
  fence_mbar_init();
}

// Producer: the next slot may be refilled once its previous stage was consumed.
__device__ __forceinline__ bool ring_reserve(const Ring& R, const RingPos& P, int* err) {
  if (P.count < R.n) return true;
  if (mbar_wait(&R.empty[P.slot], P.phase ^ 1, err)) return true;
  raise_error(err, ERR_EMPTY_WAIT);
  return false;
}

// After an error: wait (bounded in time, not cut short by the error flag) for
// the last copies into every slot, so none lands after the CTA has left.
__device__ __forceinline__ void ring_drain(const Ring& R, const RingPos& P, int* err) {
  for (int k = P.count - R.n > 0 ? P.count - R.n : 0; k < P.count; ++k)
    if (!mbar_wait(&R.full[k % R.n], (k / R.n) & 1)) raise_error(err, ERR_DRAIN);
}

// ---- GEMV --------------------------------------------------------------------
// The pointers of a GEMV phase that change from layer to layer (and, for the
// first and last layer, from step to step); everything else comes from a
// GemvParams that is the same for every layer.
struct GemvIO {
  const uint8_t* w;
  const uint16_t* norm_w;
  const float* x;
  float* x_copy;
  float* out;
  float* tap;
  uint16_t* kc;
  uint16_t* vc;
  int8_t* qtap;
  float* qstap;
  int32_t* dots;
};

__device__ __forceinline__ GemvIO gemv_io(const GemvParams& p) {
  return GemvIO{p.w, p.norm_w, p.x, p.x_copy, p.out, p.tap, p.kc, p.vc, p.qtap, p.qstap, p.dots};
}
// Work area of a GEMV phase: x (fp32, K) | [q4: int8 x (K), block scales,
// block sums] | per-warp row-block partials | warp sums + abort mark.
struct GemvLayout {
  int K, max_rb_local;
  bool q4;
  __host__ __device__ size_t qx_off() const { return 4 * (size_t)((K + 3) & ~3); }
  __host__ __device__ size_t dx_off() const { return qx_off() + (q4 ? (size_t)K : 0); }
  __host__ __device__ size_t sx_off() const { return dx_off() + (q4 ? 4 * (size_t)(K / 32) : 0); }
  __host__ __device__ size_t part_off() const { return sx_off() + (q4 ? 4 * (size_t)(K / 32) : 0); }
  __host__ __device__ size_t red_off() const {
    return part_off() + 4 * (size_t)max_rb_local * kConsumerWarps * kTileR;
  }
  __host__ __device__ size_t total() const { return red_off() + 4 * 32; }
};

struct GemvWork {
  float* xs;
  uint8_t* qx;
  float* dx;
  int* sx;
  float* part;
  float* red;
  __device__ GemvWork(uint8_t* base, const GemvLayout& L)
      : xs(reinterpret_cast<float*>(base)),
        qx(base + L.qx_off()),
        dx(reinterpret_cast<float*>(base + L.dx_off())),
        sx(reinterpret_cast<int*>(base + L.sx_off())),
        part(reinterpret_cast<float*>(base + L.part_off())),
        red(reinterpret_cast<float*>(base + L.red_off())) {}
};

// Epilogue of one finished row block (kTileR tiled rows, values v).  Returns
// the sum of squares of the rows written by a residual epilogue (0 otherwise).
template <int EPI>
__device__ __forceinline__ float gemv_epilogue(const GemvParams& p, const GemvIO& io, int rb,
                                               const float v[kTileR]) {
  const int R0 = rb * kTileR;
  if (!TLD_IN_BOUNDS(rb >= 0 && rb < p.n_rb, p.err)) return 0.f;
  if (EPI == EPI_QKV) {
    const int hd = p.hd, half = hd / 2;
    const int qrows = p.nq * hd, krows = p.nkv * hd;
    const int pos = *p.pos;
    if (!TLD_IN_BOUNDS(pos >= 0 && pos < p.max_ctx && R0 + kTileR <= qrows + 2 * krows, p.err))
      return 0.f;
    if (R0 < qrows + krows) {
      // rows (2i, 2i+1) of a head hold the two dims of RoPE pair i: rotate the pair
      const bool is_q = R0 < qrows;
      const int local = is_q ? R0 : R0 - qrows;
      const int head = local / hd, i0 = (local % hd) / 2;
      const float2* cs = p.rope + (size_t)pos * half;
#pragma unroll
      for (int pr = 0; pr < kTileR / 2; ++pr) {
        const int i = i0 + pr;
        const float a = v[2 * pr], b = v[2 * pr + 1];
        const float2 c = cs[i];
        const float ra = a * c.x - b * c.y;
        const float rb2 = a * c.y + b * c.x;
        // pair i holds dims (i, i + hd/2), or (2i, 2i + 1) with interleaved pairs
        const int e = p.rope_inter ? 2 * i : i, o = p.rope_inter ? 2 * i + 1 : i + half;
        if (is_q) {
          p.q_out[head * hd + e] = ra;
          p.q_out[head * hd + o] = rb2;
        } else {
          uint16_t* row = io.kc + kv_row_offset(p.pages, kAttnStageBytes / 4 / hd, p.nkv, p.max_ctx, hd, head, pos);
          row[e] = f32_to_bf16_bits(ra);
          row[o] = f32_to_bf16_bits(rb2);
        }
      }
    } else {
      const int local = R0 - qrows - krows;
      const int head = local / hd, j = local % hd;
      uint16_t* row = io.vc + kv_row_offset(p.pages, kAttnStageBytes / 4 / hd, p.nkv, p.max_ctx, hd, head, pos);
#pragma unroll
      for (int r = 0; r < kTileR; ++r) row[j + r] = f32_to_bf16_bits(v[r]);
    }
  } else if (EPI == EPI_RESID) {
    float ss = 0.f;
#pragma unroll
    for (int r = 0; r < kTileR; ++r) {
      const float y = __ldcg(p.resid + R0 + r) + v[r];
      io.out[R0 + r] = y;
      if (io.tap) io.tap[R0 + r] = y;
      ss = fmaf(y, y, ss);
    }
    return ss;
  } else if (EPI == EPI_LOGITS) {
#pragma unroll
    for (int r = 0; r < kTileR; ++r) io.out[R0 + r] = v[r];
  } else {  // EPI_SWIGLU: tiled rows alternate gate and up of the same output
    const int j = R0 / 2;
#pragma unroll
    for (int pr = 0; pr < kTileR / 2; ++pr) p.a_out[j + pr] = silu_f(v[2 * pr]) * v[2 * pr + 1];
  }
  return 0.f;
}

// A position in the tiled matrix, advanced without divisions.
struct TileCursor {
  int rb, kt;
  __device__ __forceinline__ void advance(int n, int ktiles) {
    kt += n;
    while (kt >= ktiles) {
      kt -= ktiles;
      ++rb;
    }
  }
  // byte offset of the tile from the matrix start
  __device__ __forceinline__ int64_t offset(const TileGeom& g) const {
    return (int64_t)rb * g.rb_bytes + (int64_t)kt * g.tile_bytes;
  }
};

// Reduce 4 per-lane row accumulators over the warp: each butterfly step keeps
// half of the rows and hands the other half to the partner lane; lane 8r ends
// with the total of row r.
__device__ __forceinline__ float warp_reduce4(const float a[4], int lane) {
  const bool h16 = lane & 16;
  const float k0 = (h16 ? a[2] : a[0]) + __shfl_xor_sync(0xffffffffu, h16 ? a[0] : a[2], 16);
  const float k1 = (h16 ? a[3] : a[1]) + __shfl_xor_sync(0xffffffffu, h16 ? a[1] : a[3], 16);
  const bool h8 = lane & 8;
  float k = (h8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

// Per-32-block absmax int8 quantization of the fp32 vector xs[K] (K % 32 == 0):
// dx = amax / 127 (fp32 divide), q = round-half-even(z / dx) clamped to +-127,
// q = 0 when dx == 0.  Eight lanes serve a block, four elements each.  The int8
// values are stored for dp4a against packed nibbles: in each group of eight,
// the even elements first, then the odd ones.  sx holds each block's sum of q.
// Correctly rounded fp32 quotient a / b from rb = RN(1/b): q = RN(a rb), the
// exact remainder r = a - b q (one FMA), then RN(q + r rb) (Markstein's
// correction, "Computation of elementary functions on the IBM RISC System/6000
// processor", 1990).  Normal operands; equal to the IEEE division on every
// case of the host check (random and next to k + 1/2 quotients).
__device__ __forceinline__ float div_rn_from_rcp(float a, float b, float rb) {
  const float q = a * rb;
  const float r = fmaf(-q, b, a);
  return fmaf(r, rb, q);
}

// Per-32-block absmax quantization of xs[0..K) * scale into the dp4a layout of
// qx (per 8 elements: the four even ones, then the four odd ones), the block
// scales dx (fp32, amax / 127) and the code sums sx; optionally also the codes in
// natural order (qtap) and the scales (qstap).  A code is round-half-even of the
// fp32 quotient z / d, clamped to +-127, formed from the block's reciprocal as
// above (three operations instead of a division).  Eight lanes a block, four
// elements a lane; each lane group takes kQuantBlocks blocks at once so that
// their shuffle and arithmetic chains overlap (measured on the int4 7B-shape
// stack: two blocks beat one, three and four, by 3.4 us per layer, as a
// 4096-element vector then keeps all sixteen warps busy).
#ifndef TLD_QUANT_BLOCKS
#define TLD_QUANT_BLOCKS 2
#endif
constexpr int kQuantBlocks = TLD_QUANT_BLOCKS;

template <bool SCALED = true>
__device__ inline void quantize_blocks(const float* xs, int K, uint8_t* qx, float* dx, int* sx,
                                       int8_t* qtap, float* qstap, int tid, int NC, float scale) {
  const int lane = tid & 31, sub = lane & 7, warp = tid >> 5;
  const int nblk = K / 32;
  constexpr int R = kQuantBlocks;
  const float r127 = 1.0f / 127.0f;
  // the trip count is the same for all lanes of a warp (the shuffles name the whole warp)
  for (int base = warp * 4 * R; base < nblk; base += (NC >> 5) * 4 * R) {
    float4 z[R];
    float amax[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int blk = base + r * 4 + (lane >> 3);
      z[r] = blk < nblk ? *reinterpret_cast<const float4*>(xs + blk * 32 + sub * 4)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      if (SCALED) {
        z[r].x *= scale;
        z[r].y *= scale;
        z[r].z *= scale;
        z[r].w *= scale;
      }
      amax[r] = fmaxf(fmaxf(fabsf(z[r].x), fabsf(z[r].y)), fmaxf(fabsf(z[r].z), fabsf(z[r].w)));
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1)
#pragma unroll
      for (int r = 0; r < R; ++r) amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], o));
    int q[R][4], sum[R];
    float dd[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float zz[4] = {z[r].x, z[r].y, z[r].z, z[r].w};
      float d;
      if (amax[r] >= 1e-30f) {
        d = div_rn_from_rcp(amax[r], 127.0f, r127);  // amax / 127
        const float rd = __frcp_rn(d);
        // no clamp needed: |z| <= amax and d >= (amax / 127)(1 - 2^-24), so
        // |z / d| <= 127 (1 + 2^-23) and its rounded fp32 quotient rounds to
        // at most 127
#pragma unroll
        for (int i = 0; i < 4; ++i) q[r][i] = __float2int_rn(div_rn_from_rcp(zz[i], d, rd));
      } else {  // a block so small that 1/d would overflow (or all zero): IEEE divisions
        d = __fdiv_rn(amax[r], 127.0f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int v = d != 0.0f ? __float2int_rn(__fdiv_rn(zz[i], d)) : 0;
          q[r][i] = v > 127 ? 127 : (v < -127 ? -127 : v);
        }
      }
      sum[r] = q[r][0] + q[r][1] + q[r][2] + q[r][3];
      dd[r] = d;
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1)
#pragma unroll
      for (int r = 0; r < R; ++r) sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], o);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int blk = base + r * 4 + (lane >> 3);
      if (blk >= nblk) continue;
      const int e = blk * 32 + sub * 4;
      // elements e..e+3 = 8g + 4h + {0,1,2,3}: evens go to bytes 8g+2h, 8g+2h+1,
      // odds to bytes 8g+4+2h, 8g+4+2h+1
      const int g8 = e & ~7, h = (e >> 2) & 1;
      *reinterpret_cast<uint16_t*>(qx + g8 + 2 * h) =
          (uint16_t)((q[r][0] & 0xff) | ((q[r][2] & 0xff) << 8));
      *reinterpret_cast<uint16_t*>(qx + g8 + 4 + 2 * h) =
          (uint16_t)((q[r][1] & 0xff) | ((q[r][3] & 0xff) << 8));
      if (sub == 0) {
        dx[blk] = dd[r];
        sx[blk] = sum[r];
      }
      if (qtap) {
#pragma unroll
        for (int i = 0; i < 4; ++i) qtap[e + i] = (int8_t)q[r][i];
        if (sub == 0) qstap[blk] = dd[r];
      }
    }
  }
}

// One warp quantizes one 32-block whose element `lane` is u, with the same
// arithmetic as quantize_blocks: the scale amax / 127, the code round-half-even
// of u / scale clamped to +-127 (0 when the scale is 0), stored at its place in
// the dp4a arrangement, and the block's code sum.
__device__ __forceinline__ void q8_block_warp(float u, int lane, uint8_t* codes, float* scale,
                                              int32_t* sum) {
  float amax = fabsf(u);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float d;
  int v;
  if (amax >= 1e-30f) {
    d = div_rn_from_rcp(amax, 127.0f, 1.0f / 127.0f);
    v = __float2int_rn(div_rn_from_rcp(u, d, __frcp_rn(d)));
  } else {
    d = __fdiv_rn(amax, 127.0f);
    v = d != 0.0f ? __float2int_rn(__fdiv_rn(u, d)) : 0;
  }
  const int q = v > 127 ? 127 : (v < -127 ? -127 : v);
  int s = q;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const int j = lane & 7;  // per 8 elements: the even ones, then the odd ones
  codes[(lane & ~7) + ((j & 1) ? 4 : 0) + (j >> 1)] = (uint8_t)(q & 0xff);
  if (lane == 0) {
    *scale = d;
    *sum = s;
  }
}

// Publication of an output vector's int8 quantization (see QVec) after this
// CTA wrote its elements [e0, e1) of v.  Every writer has passed a CTA barrier
// after its stores before this call.  One warp per block this CTA touched:
// lane 0 adds the CTA's element count to the block's counter; the CTA that
// brings it to a multiple of 32 wrote the block's last element and quantizes
// the block from L2 (times the norm weight, if any).
__device__ __forceinline__ void q8_publish(const QVec& q, const float* v, int e0, int e1, int warp,
                                           int lane, int nwarps, int* err) {
  const int b0 = e0 >> 5, b1 = (e1 + 31) >> 5;
  for (int blk = b0 + warp; blk < b1; blk += nwarps) {
    if (!TLD_IN_BOUNDS(blk >= 0 && blk < q.K / 32, err)) break;
    int last = 0;
    if (lane == 0) {
      __threadfence();  // this CTA's elements before its count
      const int lo = e0 > (blk << 5) ? e0 : (blk << 5);
      const int hi = e1 < ((blk + 1) << 5) ? e1 : ((blk + 1) << 5);
      const unsigned n = (unsigned)(hi - lo);
      const unsigned old = atomicAdd(q.cnt + blk, n);
      last = ((old + n) & 31u) == 0u;
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) continue;
    __threadfence();  // the other CTAs' elements, fenced before their counts
    const int e = (blk << 5) + lane;
    float u = __ldcg(v + e);
    if (q.w) u *= __uint_as_float((uint32_t)q.w[e] << 16);
    q8_block_warp(u, lane, q.codes + (blk << 5), q.scale + blk, q.sum + blk);
  }
}

// Four-way byte dot with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Integer dot of one 32-block: packed nibbles (q + 8) against the arranged
// int8 activations, minus 8 * (sum of the activations).  The low nibbles are
// masked in place; the high nibbles are masked without a shift, so their bytes
// hold 16 x the nibble (unsigned) and their dot is 16 x theirs, divided out
// exactly at the end.
__device__ __forceinline__ int q4_block_dot(const uint4 w, const uint4 x0, const uint4 x1, int sx) {
  constexpr uint32_t M = 0x0F0F0F0Fu;
  int lo = 0, hi = 0;
  lo = __dp4a((int)(w.x & M), (int)x0.x, lo);
  hi = dp4a_us(w.x & ~M, x0.y, hi);
  lo = __dp4a((int)(w.y & M), (int)x0.z, lo);
  hi = dp4a_us(w.y & ~M, x0.w, hi);
  lo = __dp4a((int)(w.z & M), (int)x1.x, lo);
  hi = dp4a_us(w.z & ~M, x1.y, hi);
  lo = __dp4a((int)(w.w & M), (int)x1.z, lo);
  hi = dp4a_us(w.w & ~M, x1.w, hi);
  return lo + (hi >> 4) - 8 * sx;
}

// One stage as `copies` bulk copies of about equal size on the same barrier:
// several copies in flight move a stage into shared memory faster than one
// large copy (measured on the 7B-shape stacks: four for bf16 stages, +1.7 %
// over one; eight for int4 stages, +2.7 % over four, where eight slow bf16).
template <int COPIES>
__device__ __forceinline__ void bulk_g2s_split_n(uint8_t* dst, const uint8_t* src, uint32_t bytes,
                                                 uint64_t* bar, uint64_t pol) {
  const uint32_t part = (bytes / COPIES) & ~15u;
  uint32_t o = 0;
  if (part > 0)
#pragma unroll
    for (int k = 0; k < COPIES - 1; ++k, o += part) bulk_g2s_hint(dst + o, src + o, part, bar, pol);
  bulk_g2s_hint(dst + o, src + o, bytes - o, bar, pol);
}
__device__ __forceinline__ void bulk_g2s_split(uint8_t* dst, const uint8_t* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t pol, int copies) {
  if (copies == kCopiesPerStageQ4)
    bulk_g2s_split_n<kCopiesPerStageQ4>(dst, src, bytes, bar, pol);
  else
    bulk_g2s_split_n<kCopiesPerStage>(dst, src, bytes, bar, pol);
}

// Producer of a GEMV phase: this CTA's slab, whole row blocks [rb0, rb1).
__device__ __forceinline__ void gemv_produce(const GemvParams& p, const uint8_t* w, const Ring& R,
                                             RingPos& P, int rb0, int rb1, uint64_t pol) {
  const TileGeom& geo = p.geo;
  const int nloc = (rb1 - rb0) * geo.ktiles;
  const int nst = (nloc + kStageTiles - 1) / kStageTiles;
  TileCursor cur{rb0, 0};
  const int64_t end_off = (int64_t)rb1 * geo.rb_bytes;
  for (int s = 0; s < nst; ++s) {
    if (!ring_reserve(R, P, p.err)) return;
    const int64_t oa = cur.offset(geo);
    cur.advance(kStageTiles, geo.ktiles);
    const int64_t ob = (s == nst - 1) ? end_off : cur.offset(geo);
    if (!TLD_IN_BOUNDS(oa >= 0 && ob > oa && ob <= (int64_t)p.n_rb * geo.rb_bytes &&
                           ob - oa <= R.slot_bytes, p.err))
      return;
    const uint32_t bytes = (uint32_t)(ob - oa);
    mbar_arrive_expect_tx(&R.full[P.slot], bytes);
    bulk_g2s_split(R.slot(P.slot), w + oa, bytes, &R.full[P.slot], pol, geo.copies);
    P.next(R.n);
  }
}

// L2 prefetch of this CTA index's share of the next kernel (see L2Ahead).
template <int HD>
__device__ void l2_ahead_kv(const L2Ahead& a, int b);

__device__ __forceinline__ void l2_ahead(const L2Ahead& a, int b) {
  if (!a.base || b >= a.grid) return;
  if (a.kv) {
    if (a.hd == 64) l2_ahead_kv<64>(a, b);
    else l2_ahead_kv<128>(a, b);
    return;
  }
  const int64_t r0 = split_begin(a.n_units, a.grid, b), r1 = split_begin(a.n_units, a.grid, b + 1);
  int64_t left = (r1 - r0) * a.unit_bytes;
  if (left > a.cap) left = a.cap;
  // 16-byte aligned start (the buffers themselves are)
  const int64_t start = r0 * a.unit_bytes, lead = start & 15;
  const uint8_t* src = a.base + (start - lead);
  left = (left + lead) & ~(int64_t)15;
  if (!TLD_IN_BOUNDS(start - lead + left <= (int64_t)a.n_units * a.unit_bytes, nullptr)) return;
  for (int64_t o = 0; o < left; o += kStageBytes) {
    const int64_t n = left - o < kStageBytes ? left - o : kStageBytes;
    bulk_prefetch_l2(src + o, (uint32_t)n);
  }
}

// Consumer work of a GEMV phase that does not depend on its input vector:
// the RMSNorm weights (static) go to xs as fp32; the partials are cleared.
template <int PRO>
__device__ __forceinline__ void gemv_pre(const GemvParams& p, const uint16_t* norm_w,
                                         const GemvWork& W, int tid) {
  const int K4 = p.geo.K / 4;
  if (PRO == PRO_NORM) {
    const uint2* w4 = reinterpret_cast<const uint2*>(norm_w);
    for (int k4 = tid; k4 < K4; k4 += kNC) {
      const uint2 wb = w4[k4];
      reinterpret_cast<float4*>(W.xs)[k4] =
          make_float4(bf16lo(wb.x), bf16hi(wb.x), bf16lo(wb.y), bf16hi(wb.y));
    }
  }
  for (int i = tid; i < p.max_rb_local * kConsumerWarps * kTileR; i += kNC) W.part[i] = 0.f;
  if (tid == 0) W.red[kConsumerWarps] = 0.f;
}

// Consumer part of a GEMV phase once its input vector is ready: the prologue
// (input, RMSNorm, quantisation), the streaming loop over this CTA's tiles and
// the row-block epilogue.  Returns false if a wait ran out.
template <int PRO, int EPI, bool Q4>
__device__ __forceinline__ bool gemv_main(const GemvParams& p, const GemvIO& io, const GemvWork& W,
                                          const Ring& R, RingPos& P, int rb0, int rb1, int tid,
                                          bool first_cta) {
  const TileGeom& geo = p.geo;
  const int K = geo.K, K4 = K / 4;
  const int warp = tid >> 5, lane = tid & 31;
  const int nrb = rb1 - rb0;
  const int nloc = nrb * geo.ktiles;
  const int nst = (nloc + kStageTiles - 1) / kStageTiles;
  float* xs = W.xs;
  // q4 with a published input: the codes, not the vector, are read below
  const bool qin = Q4 && p.qin.codes != nullptr;
  if (!qin) {
    // the input vector was written by another phase: read it from L2
    const float4* x4 = reinterpret_cast<const float4*>(io.x);
    float ss = 0.f;
    constexpr int PB = 12;  // loads in flight per thread: K up to 12288 in one round trip
    for (int base = tid; base < K4; base += kNC * PB) {
      float4 v[PB];
#pragma unroll
      for (int u = 0; u < PB; ++u)
        if (base + u * kNC < K4) v[u] = __ldcg(x4 + base + u * kNC);
#pragma unroll
      for (int u = 0; u < PB; ++u) {
        const int k4 = base + u * kNC;
        if (k4 >= K4) continue;
        if (PRO == PRO_NORM) {
          ss += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
          float4 w = reinterpret_cast<float4*>(xs)[k4];
          w.x *= v[u].x;
          w.y *= v[u].y;
          w.z *= v[u].z;
          w.w *= v[u].w;
          reinterpret_cast<float4*>(xs)[k4] = w;
        } else {
          reinterpret_cast<float4*>(xs)[k4] = v[u];
        }
      }
    }
    if (PRO == PRO_NORM) {
      ss = warp_sum(ss);
      if (lane == 0) W.red[warp] = ss;
    }
  }
  if (io.x_copy && first_cta) {
    for (int k = tid; k < K; k += kNC) io.x_copy[k] = __ldcg(io.x + k);
  }
  if (p.pos_advance && first_cta && tid == 0) atomicAdd(p.pos_advance, 1);
  if (qin) {
    // The producer has finished (griddepcontrol.wait): clear its per-block
    // counts for the next round, take the 1/rms from its per-CTA sums of
    // squares (added in CTA order, the same in every CTA), and copy the codes,
    // scales (times 1/rms) and sums into shared memory.
    if (first_cta && p.qin.cnt)
      for (int i = tid; i < K / 32; i += kNC) p.qin.cnt[i] = 0u;
    // everything in one round trip: codes and sums to shared memory, the scales
    // and the producers' sums of squares (into xs, unused here) to be scaled
    const uint4* c4 = reinterpret_cast<const uint4*>(p.qin.codes);
    for (int i = tid; i < K / 16; i += kNC) reinterpret_cast<uint4*>(W.qx)[i] = __ldcg(c4 + i);
    for (int i = tid; i < K / 32; i += kNC) {
      W.dx[i] = __ldcg(p.qin.scale + i);
      W.sx[i] = __ldcg(p.qin.sum + i);
    }
    const int np = PRO == PRO_NORM ? p.qin.n_part : 0;
    for (int c = tid; c < np; c += kNC) xs[c] = __ldcg(p.qin.part + c);
    named_barrier(1, kNC);
    if (PRO == PRO_NORM) {
      float s = 0.f;
      for (int c = lane; c < np; c += 32) s += xs[c];
      s = warp_sum(s);  // the same order, so the same value, in every warp and CTA
      const float rn = 1.0f / sqrtf(s / (float)K + p.eps);
      for (int i = tid; i < K / 32; i += kNC) W.dx[i] *= rn;
    }
    if (first_cta && io.qstap)
      for (int i = tid; i < K / 32; i += kNC) io.qstap[i] = W.dx[i];
  }
  named_barrier(1, kNC);
  if (qin && first_cta && io.qtap) {
    for (int e = tid; e < K; e += kNC)
      io.qtap[e] = (int8_t)W.qx[(e & ~7) + ((e & 1) ? 4 : 0) + ((e & 7) >> 1)];
  }

  // RMSNorm is a per-vector scale 1/sqrt(mean(x^2)+eps).  bf16 weights: the
  // projection runs on x*w and the scale multiplies the finished rows.  q4
  // weights: the normalised vector itself is quantised, so it is scaled first.
  float rnorm = 1.f;
  if (PRO == PRO_NORM && !qin) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += W.red[w];
    rnorm = 1.0f / sqrtf(tot / (float)K + p.eps);
  }
  if (Q4 && !qin) {
    // the normalised vector itself is quantised: the codes carry the RMS scale
    if (PRO == PRO_NORM)
      quantize_blocks<true>(xs, K, W.qx, W.dx, W.sx, first_cta ? io.qtap : nullptr, io.qstap, tid,
                            kNC, rnorm);
    else  // the plain input: no scale
      quantize_blocks<false>(xs, K, W.qx, W.dx, W.sx, first_cta ? io.qtap : nullptr, io.qstap, tid,
                             kNC, 1.f);
    rnorm = 1.f;
    named_barrier(1, kNC);
  }

  int cur_rb = -1;
  float acc[kTileR];
#pragma unroll
  for (int r = 0; r < kTileR; ++r) acc[r] = 0.f;
  bool ok = true;
  // cursors: the first tile of the current stage and this warp's two tiles in it
  TileCursor st_cur{rb0, 0};
  TileCursor my[kTilesPerWarp];
#pragma unroll
  for (int j = 0; j < kTilesPerWarp; ++j) {
    my[j] = st_cur;
    my[j].advance(warp + j * kConsumerWarps, geo.ktiles);
  }
  // bf16: lane owns columns [8 lane, 8 lane + 8) of a tile; q4: lane owns block `lane`
  const int c = Q4 ? lane * 32 : lane * 8;
  for (int s = 0; s < nst; ++s) {
    // After a timed-out wait the warp stops waiting but keeps the same control
    // flow, so that every named barrier below is still reached by all warps.
    if (ok && !mbar_wait(&R.full[P.slot], P.phase, p.err)) {
      raise_error(p.err, ERR_FULL_WAIT);
      ok = false;
    }
    if (s == 0 && tid == 0) tl_mark_max(p.tl, 4);
    // Copy this warp's tiles into registers and hand the slot back at once, so
    // the next bulk copy is in flight while the arithmetic runs.
    uint4 wv[kTilesPerWarp][kTileR];
    uint2 scl[kTilesPerWarp];
    const int64_t st_off = st_cur.offset(geo);
#pragma unroll
    for (int j = 0; j < kTilesPerWarp; ++j) {
      const int li = s * kStageTiles + warp + j * kConsumerWarps;
      const int kw = (my[j].kt == geo.ktiles - 1) ? geo.kw_last : geo.tile_k;
      if (li < nloc && c < kw &&
          TLD_IN_BOUNDS(my[j].offset(geo) - st_off >= 0 &&
                            my[j].offset(geo) - st_off + geo.tile_bytes <= R.slot_bytes, p.err)) {
        const uint8_t* tp = R.slot(P.slot) + (my[j].offset(geo) - st_off);
        if (Q4) {
#pragma unroll
          for (int r = 0; r < kTileR; ++r)
            wv[j][r] = *reinterpret_cast<const uint4*>(tp + (size_t)r * (kw / 2) + lane * 16);
          scl[j] = *reinterpret_cast<const uint2*>(tp + (size_t)kTileR * (kw / 2) + lane * 8);
        } else {
#pragma unroll
          for (int r = 0; r < kTileR; ++r)
            wv[j][r] = *reinterpret_cast<const uint4*>(tp + ((size_t)r * kw + c) * 2);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[P.slot]);
#pragma unroll
    for (int j = 0; j < kTilesPerWarp; ++j) {
      const int li = s * kStageTiles + warp + j * kConsumerWarps;
      if (li >= nloc) continue;
      const int rb = my[j].rb, kt = my[j].kt;
      if (rb != cur_rb) {
        if (cur_rb >= 0) {
          const float v = warp_reduce4(acc, lane);
          if ((lane & 7) == 0)
            W.part[((cur_rb - rb0) * kConsumerWarps + warp) * kTileR + (lane >> 3)] = v;
        }
        cur_rb = rb;
#pragma unroll
        for (int r = 0; r < kTileR; ++r) acc[r] = 0.f;
      }
      const int kw = (kt == geo.ktiles - 1) ? geo.kw_last : geo.tile_k;
      if (c >= kw) continue;
      if (Q4) {
        const int blk = kt * (kTileKQ4 / 32) + lane;
        const uint4 x0 = *reinterpret_cast<const uint4*>(W.qx + blk * 32);
        const uint4 x1 = *reinterpret_cast<const uint4*>(W.qx + blk * 32 + 16);
        const float dxb = W.dx[blk];
        const int sxb = W.sx[blk];
        const uint32_t sc2[2] = {scl[j].x, scl[j].y};
#pragma unroll
        for (int r = 0; r < kTileR; ++r) {
          const int idot = q4_block_dot(wv[j][r], x0, x1, sxb);
          const uint16_t hb = (uint16_t)(r & 1 ? sc2[r >> 1] >> 16 : sc2[r >> 1] & 0xffff);
          const float sw = __half2float(__ushort_as_half(hb));
          acc[r] = fmaf(sw * dxb, (float)idot, acc[r]);
          if (io.dots) io.dots[(size_t)(rb * kTileR + r) * (K / 32) + blk] = idot;
        }
      } else {
        const float4 xa = *reinterpret_cast<const float4*>(xs + kt * kTileK + c);
        const float4 xb = *reinterpret_cast<const float4*>(xs + kt * kTileK + c + 4);
#pragma unroll
        for (int r = 0; r < kTileR; ++r) {
          float a = acc[r];
          a = fmaf(bf16lo(wv[j][r].x), xa.x, a);
          a = fmaf(bf16hi(wv[j][r].x), xa.y, a);
          a = fmaf(bf16lo(wv[j][r].y), xa.z, a);
          a = fmaf(bf16hi(wv[j][r].y), xa.w, a);
          a = fmaf(bf16lo(wv[j][r].z), xb.x, a);
          a = fmaf(bf16hi(wv[j][r].z), xb.y, a);
          a = fmaf(bf16lo(wv[j][r].w), xb.z, a);
          a = fmaf(bf16hi(wv[j][r].w), xb.w, a);
          acc[r] = a;
        }
      }
    }
    st_cur.advance(kStageTiles, geo.ktiles);
#pragma unroll
    for (int j = 0; j < kTilesPerWarp; ++j) my[j].advance(kStageTiles, geo.ktiles);
    P.next(R.n);
  }
  if (cur_rb >= 0) {
    const float v = warp_reduce4(acc, lane);
    if ((lane & 7) == 0)
      W.part[((cur_rb - rb0) * kConsumerWarps + warp) * kTileR + (lane >> 3)] = v;
  }
  if (!ok && lane == 0) W.red[kConsumerWarps] = 1.f;  // abort mark
  named_barrier(1, kNC);
  if (tid == 0) {
    tl_mark_min(p.tl, 5);
    tl_mark_max(p.tl, 6);
  }
  if (W.red[kConsumerWarps] != 0.f) return false;

  // ---- finish this CTA's row blocks (sum over warps in warp order) ------------
  // one thread per row, four neighbouring lanes per row block; the lane of
  // row 0 gathers the block's four rows and runs its epilogue
  static_assert(kTileR == 4, "four rows per row block");
  const int n4 = nrb * kTileR;
  float ssq = 0.f;  // sum of squares of the residual rows this thread wrote
  for (int base = 0; base < n4; base += kNC) {  // the same trip count in every warp
    const int t = base + tid;
    float sum = 0.f;
    if (t < n4) {
      const int j = t >> 2, r = t & 3;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) sum += W.part[(j * kConsumerWarps + w) * kTileR + r];
      sum *= rnorm;
    }
    float v[kTileR];
#pragma unroll
    for (int r = 0; r < kTileR; ++r) v[r] = __shfl_sync(0xffffffffu, sum, (lane & ~3) + r);
    if (t < n4 && (t & 3) == 0) ssq += gemv_epilogue<EPI>(p, io, rb0 + (t >> 2), v);
  }
  if (Q4 && (EPI == EPI_RESID || EPI == EPI_SWIGLU) && p.qout.codes) {
    // publish the int8 quantization of this GEMV's output for the next GEMV
    // (the CTA barrier below orders every thread's stores before the fence that
    // precedes each block count)
    if (p.qout.part) {
      ssq = warp_sum(ssq);
      if (lane == 0) W.red[warp] = ssq;
    }
    named_barrier(1, kNC);
    if (p.qout.part && tid == 0) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) tot += W.red[w];
      p.qout.part[blockIdx.x] = tot;
    }
    const int per = EPI == EPI_SWIGLU ? kTileR / 2 : kTileR;  // outputs per row block
    q8_publish(p.qout, EPI == EPI_SWIGLU ? p.a_out : io.out, rb0 * per, rb1 * per, warp, lane,
               kConsumerWarps, p.err);
  }
  return true;
}

constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// ---- attention ---------------------------------------------------------------
// One unit = one chunk of CH cached positions of one KV head (its K rows, then
// its V rows, 16 KB each).  The grid splits the units of all KV heads evenly;
// every CTA serves all G query heads of the KV heads it touches, so each K/V
// byte is read once.  Within a CTA the consumer warps take interleaved
// positions of each chunk and keep a running (max, sum, acc) per query head;
// warps are merged at the end of each head segment.  A head cut between CTAs
// is merged in one of two ways: (global) each CTA leaves a record in global
// memory and the last of the head's CTAs to finish merges them; (cluster) the
// grid is one thread-block cluster per KV head, its CTAs split that head's
// chunks, leave their records in their own shared memory, and every CTA of
// the cluster merges a slice of the head's outputs through distributed shared
// memory.

// Work area of an attention phase: per-warp states | this CTA's record
// (cluster merge) | merge scratch (global merge).
struct AttnLayout {
  int hd, G, nw = kConsumerWarps;  // nw: consumer warps of the kernel
  bool ring_ws = false;            // per-warp states in the drained ring (cluster kernel)
  __host__ __device__ size_t rec_off() const { return ring_ws ? 0 : 4 * (size_t)nw * G * (hd + 2); }
  __host__ __device__ size_t merge_off() const { return rec_off() + 4 * (size_t)G * (hd + 2); }
  // the record offsets of the splits of two heads, then the heads to merge
  __host__ __device__ size_t push_off() const { return merge_off() + 4 * (size_t)2 * kMaxSplits + 16; }
  // cluster merge: the slice of every CTA's record this CTA merges, pushed by
  // the other CTAs: [C][slice] values, then [C][G] (max, sum); at most
  // G*hd + C*(32 + 2G) floats for any cluster size C
  __host__ __device__ size_t total() const {
    return push_off() + 4 * ((size_t)G * hd + (size_t)kMaxCluster * (32 + 2 * G));
  }
};

// This CTA's share of the attention units at KV length n.
struct AttnSplit {
  int n, cph, U, u0, u1, nu;
};

template <int HD>
__device__ __forceinline__ AttnSplit attn_split(int pos, int nkv, int b, int nb) {
  constexpr int CH = kAttnStageBytes / 2 / (HD * 2);
  AttnSplit S;
  S.n = pos + 1;
  S.cph = (S.n + CH - 1) / CH;
  S.U = nkv * S.cph;
  S.u0 = split_begin32(S.U, nb, b);
  S.u1 = split_begin32(S.U, nb, b + 1);
  S.nu = S.u1 - S.u0;
  return S;
}

// Cluster split: cluster g = b / C serves KV head g; its CTA of rank r takes a
// contiguous share of that head's chunks.
template <int HD>
__device__ __forceinline__ AttnSplit attn_split_cluster(int pos, int nkv, int b, int C) {
  constexpr int CH = kAttnStageBytes / 2 / (HD * 2);
  AttnSplit S;
  S.n = pos + 1;
  S.cph = (S.n + CH - 1) / CH;
  S.U = nkv * S.cph;
  const int g = b / C, r = b - g * C;
  S.u0 = g * S.cph + split_begin32(S.cph, C, r);
  S.u1 = g * S.cph + split_begin32(S.cph, C, r + 1);
  S.nu = S.u1 - S.u0;
  return S;
}

template <int HD>
__device__ void l2_ahead_kv(const L2Ahead& a, int b) {
  constexpr int CH = kAttnStageBytes / 2 / (HD * 2);
  const AttnSplit S = a.cluster ? attn_split_cluster<HD>(*a.pos, a.nkv, b, a.cluster)
                                : attn_split<HD>(*a.pos, a.nkv, b, a.grid);
  int left = a.cap;
  int u = S.u0;
  if (a.pages) {  // one chunk (page) at a time
    for (; u < S.u1 && left > 0; ++u) {
      const int g = u / S.cph, c = u - g * S.cph;
      const int rows = min(CH, S.n - c * CH);
      int bytes = rows * HD * 2;
      if (bytes > left / 2) bytes = left / 2;
      const size_t off = (size_t)kv_row_offset(a.pages, CH, a.nkv, a.max_ctx, HD, g, c * CH) * 2;
      const uint32_t n = (uint32_t)bytes & ~15u;
      if (n) {
        bulk_prefetch_l2(a.base + off, n);
        bulk_prefetch_l2(a.vbase + off, n);
      }
      left -= 2 * bytes;
    }
    return;
  }
  while (u < S.u1 && left > 0) {
    // one head segment: its chunks are contiguous in K and in V
    const int g = u / S.cph, c0 = u - g * S.cph;
    const int c1 = min(S.cph, c0 + (S.u1 - u));
    const int rows = min(c1 * CH, S.n) - c0 * CH;
    int bytes = rows * HD * 2;
    if (bytes > left / 2) bytes = left / 2;
    const size_t off = ((size_t)g * a.max_ctx + (size_t)c0 * CH) * HD * 2;
    for (int o = 0; o < bytes; o += kStageBytes) {
      const uint32_t n = (uint32_t)min(bytes - o, kStageBytes) & ~15u;
      bulk_prefetch_l2(a.base + off + o, n);
      bulk_prefetch_l2(a.vbase + off + o, n);
    }
    left -= 2 * bytes;
    u += c1 - c0;
  }
}

// DL consecutive bf16 of one cached row, as raw bits (DL = 2 or 4).
template <int DL>
struct RowSlice {
  uint32_t w[DL / 2];
  __device__ __forceinline__ void load(const uint8_t* p) {
    if (DL == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      w[0] = v.x;
      w[DL / 2 - 1] = v.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t*>(p);
    }
  }
  __device__ __forceinline__ void unpack(float* f) const {
#pragma unroll
    for (int i = 0; i < DL / 2; ++i) {
      f[2 * i] = bf16lo(w[i]);
      f[2 * i + 1] = bf16hi(w[i]);
    }
  }
};

// Producer of an attention phase: this CTA's chunks.  wait_pos() is called
// once before the first chunk that holds the row appended by this step's QKV
// phase (the other rows were written by earlier steps).
template <int HD, class WaitPos>
__device__ __forceinline__ void attn_produce(const AttnParams& p, const uint16_t* kc,
                                             const uint16_t* vc, const Ring& R, RingPos& P,
                                             const AttnSplit& S, uint64_t pol, WaitPos&& wait_pos) {
  constexpr int CH = kAttnStageBytes / 2 / (HD * 2);
  bool waited = false;
  int g = S.u0 / S.cph, c = S.u0 - g * S.cph;
  for (int s = 0; s < S.nu; ++s) {
    if (!ring_reserve(R, P, p.err)) return;
    const int rows = min(CH, S.n - c * CH);
    if (!TLD_IN_BOUNDS(g >= 0 && g < p.nkv && rows > 0 && c * CH + rows <= p.max_ctx &&
                           2 * kAttnStageBytes / 2 <= R.slot_bytes, p.err))
      return;
    if (c == S.cph - 1 && !waited) {
      wait_pos();
      waited = true;
    }
    const size_t off = (size_t)kv_row_offset(p.pages, CH, p.nkv, p.max_ctx, HD, g, c * CH);
    const uint32_t bytes = (uint32_t)rows * HD * 2;
    mbar_arrive_expect_tx(&R.full[P.slot], 2 * bytes);
    uint8_t* dst = R.slot(P.slot);
    bulk_g2s_hint(dst, kc + off, bytes, &R.full[P.slot], pol);
    bulk_g2s_hint(dst + kAttnStageBytes / 2, vc + off, bytes, &R.full[P.slot], pol);
    if (++c == S.cph) {
      c = 0;
      ++g;
    }
    P.next(R.n);
  }
}

// The cluster merge of the attention + head-projection kernel: instead of two
// cluster-wide barriers (which the producer, still streaming the projection's
// weights, cannot join), three mbarriers per CTA that the consumers of every
// CTA arrive on remotely: records ready, o_g pushed, records read.  og is this
// CTA's copy of the group's merged output, filled by every CTA of the cluster.
struct ClusterXchg {
  float* og;       // [G * HD]
  uint64_t* bars;  // [3]: records ready, og complete, records read (C arrivals each)
};

// Consumer part of an attention phase (q must be ready).  Returns false if a
// wait ran out.
template <int HD, int G, bool CL = false, int NW = kConsumerWarps, bool XG = false>
__device__ __forceinline__ bool attn_main(const AttnParams& p, uint8_t* work, const Ring& R, RingPos& P,
                          const AttnSplit& S, int b, int nb, int tid,
                          const ClusterXchg* xg = nullptr) {
  constexpr int CH = kAttnStageBytes / 2 / (HD * 2);  // positions per chunk (16 KB of K)
  constexpr int NC = NW * 32;                          // consumer threads
  constexpr int PW = CH / NW;                          // positions per warp per chunk
  constexpr int SUB = 4;                               // positions per online-softmax update
  constexpr int DL = HD / 32;                          // dims per lane
  // Fast form (PW * G <= 32 partial dots per lane): one reduce-scatter
  // butterfly sums all of a chunk's dots, leaving lane l the total of dot
  // number (l >> SH) & (V - 1), dot v = (head gg, position i) at v = gg*PW + i;
  // each lane then runs the online softmax for its own (position, head): the
  // reference max of head gg is shared by the lanes of that head, the sum of
  // the weights is kept per (position, head) and summed over the positions
  // when the segment ends.
  constexpr int V = PW * G;
  constexpr bool FAST = V <= 32;
  constexpr int LV = FAST ? ilog2(V) : 0, LPW = ilog2(PW), SH = 5 - LV;
  const int warp = tid >> 5, lane = tid & 31;
  // The cluster kernel (no XG) ends its only head segment after its last
  // stage: its per-warp states go into the drained ring, so the work area need
  // not hold them and the ring keeps its stages.
  constexpr bool RING_WS = CL && !XG;
  const AttnLayout AL{HD, G, NW, RING_WS};
  float* ws = reinterpret_cast<float*>(RING_WS ? R.stages : work);  // [warp][G][HD+2]
  float* crec = reinterpret_cast<float*>(work + AL.rec_off());  // [G][HD+2]
  const int n = S.n, cph = S.cph, U = S.U, u0 = S.u0, u1 = S.u1, nu = S.nu;
  float m[G], l[G], acc[G][DL];
  float m_mine = -INFINITY, l_mine = 0.f;  // fast form: head's reference max, slot's sum
  const int my_v = (lane >> SH) & (V - 1), my_i = my_v % PW;
  int cur_g = -1, seg_idx = 0;
  auto reset = [&]() {
    m_mine = -INFINITY;
    l_mine = 0.f;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      m[gg] = -INFINITY;
      l[gg] = 0.f;
#pragma unroll
      for (int j = 0; j < DL; ++j) acc[gg][j] = 0.f;
    }
  };
  float qr[G][DL];
  // Ends the segment of KV head g: merge the warps' states; a head this CTA
  // covered whole is normalised into o, a split head leaves a partial record
  // (acc, m, l), merged after the loop by the last CTA of the head to finish.
  int split_heads[2] = {-1, -1};
  // Cluster merge by pushing (no XG): element e of the group's G*HD outputs is
  // merged by the CTA owning its 32-block (rank order of whole blocks); each
  // CTA writes its (acc) for e into that CTA's slot of the pushed slices, and
  // its (max, sum) of every head into every CTA.
  const int cC = CL ? p.cluster : 1, cr_rank = CL ? (int)cluster_rank() : 0;
  constexpr int NBLK = G * HD / 32;
  const int MS = 32 * ((NBLK + cC - 1) / cC);  // largest slice
  float* pv = reinterpret_cast<float*>(work + AL.push_off());  // [C][MS]
  float* pml = pv + (size_t)cC * MS;                                               // [C][G][2]
  auto push_record = [&](int gg, int j, float A, float M, float Ls) {
    const int e = gg * HD + j, rr = split_owner32(NBLK, cC, e >> 5);
    const int k = e - 32 * split_begin32(NBLK, cC, rr);
    if (!TLD_IN_BOUNDS(rr >= 0 && rr < cC && k >= 0 && k < MS, p.err)) return;
    dsmem_st(dsmem_addr(pv + (size_t)cr_rank * MS + k, (uint32_t)rr), A);
    if (j == 0)
      for (int c2 = 0; c2 < cC; ++c2) {
        const float* ml = pml + ((size_t)cr_rank * G + gg) * 2;
        dsmem_st(dsmem_addr(ml, (uint32_t)c2), M);
        dsmem_st(dsmem_addr(ml + 1, (uint32_t)c2), Ls);
      }
  };
  if (CL && !XG) cluster_wait();  // every CTA of the cluster is running before the first push
  auto end_segment = [&](int g) {
    if (FAST) {
      float lsum = l_mine;  // over the positions of this lane's head
#pragma unroll
      for (int bt = 0; bt < LPW; ++bt) lsum += __shfl_xor_sync(0xffffffffu, lsum, 1 << (SH + bt));
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        m[gg] = __shfl_sync(0xffffffffu, m_mine, (gg * PW) << SH);
        l[gg] = __shfl_sync(0xffffffffu, lsum, (gg * PW) << SH);
      }
    }
    if (RING_WS) {
      // every warp is past its last stage (the bulk copies into the ring are
      // complete and read) before the ring is written as plain shared memory
      named_barrier(1, NC);
      fence_proxy_async_shared();
      if (!TLD_IN_BOUNDS((size_t)NW * G * (HD + 2) * 4 <= (size_t)R.n * R.slot_bytes, p.err)) return;
    }
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
    const int64_t h0 = (int64_t)g * cph, h1 = h0 + cph;
    const bool whole = !CL && h0 >= u0 && h1 <= u1;
    if (!CL && !whole) split_heads[seg_idx == 0 ? 0 : 1] = g;
    float* rec = p.part + ((size_t)b * 2 + (seg_idx == 0 ? 0 : 1)) * G * (HD + 4);
    for (int i = tid; i < G * HD; i += NC) {
      const int gg = i / HD, j = i % HD;
      float M = -INFINITY;
      for (int w = 0; w < NW; ++w) M = fmaxf(M, ws[(w * G + gg) * (HD + 2) + HD]);
      float A = 0.f, Ls = 0.f;
      for (int w = 0; w < NW; ++w) {
        const float* wr = ws + (w * G + gg) * (HD + 2);
        const float e = (wr[HD] == -INFINITY) ? 0.f : expf(wr[HD] - M);
        A += wr[j] * e;
        Ls += wr[HD + 1] * e;
      }
      if (CL && !XG) {  // into the shared memory of the CTA that merges element (gg, j)
        push_record(gg, j, A, M, Ls);
      } else if (CL) {  // this CTA's record, in its own shared memory
        float* cr = crec + gg * (HD + 2);
        cr[j] = A;
        if (j == 0) {
          cr[HD] = M;
          cr[HD + 1] = Ls;
        }
      } else if (whole) {
        const size_t oi = (size_t)(g * G + gg) * HD + j;
        p.o[oi] = A / Ls;
        if (p.qout.codes)  // the int8 input of the o-proj, one block per warp
          q8_block_warp(A / Ls, tid & 31, p.qout.codes + (oi & ~(size_t)31),
                        p.qout.scale + (oi >> 5), p.qout.sum + (oi >> 5));
      } else {
        rec[gg * (HD + 4) + j] = A;
        if (j == 0) {
          rec[gg * (HD + 4) + HD] = M;
          rec[gg * (HD + 4) + HD + 1] = Ls;
        }
      }
    }
    // The records are released to the other CTAs by the ticket below: this
    // barrier orders every thread's writes before thread 0's gpu-scope release.
    named_barrier(1, NC);
    ++seg_idx;
  };

  reset();
  if (CL && nu == 0) {  // no chunk of the head: an empty record
    if (XG) {
      for (int i = tid; i < G * (HD + 2); i += NC) crec[i] = (i % (HD + 2) == HD) ? -INFINITY : 0.f;
    } else {
      for (int i = tid; i < G * HD; i += NC) push_record(i / HD, i % HD, 0.f, -INFINITY, 0.f);
    }
  }
  bool ok = true;
  int g = u0 / cph, c = u0 - g * cph;
  for (int s = 0; s < nu; ++s) {
    if (g != cur_g) {
      if (cur_g >= 0) {
        end_segment(cur_g);
        reset();
      }
      cur_g = g;
#pragma unroll
      for (int gg = 0; gg < G; ++gg)
#pragma unroll
        for (int j = 0; j < DL; ++j) qr[gg][j] = __ldcg(p.q + (size_t)(g * G + gg) * HD + lane * DL + j) * p.scale;
    }
    if (ok && !mbar_wait(&R.full[P.slot], P.phase, p.err)) {
      raise_error(p.err, ERR_FULL_WAIT);
      ok = false;  // keep the control flow (segment barriers) uniform
    }
    if (s == 0 && tid == 0) tl_mark_max(p.tl, 4);
    const int rows = min(CH, n - c * CH);
    const uint8_t* kb = R.slot(P.slot);
    const uint8_t* vb = kb + kAttnStageBytes / 2;
    // This warp's K and V row slices into registers, then the slot goes back.
    RowSlice<DL> kr[PW], vr[PW];
#pragma unroll
    for (int i = 0; i < PW; ++i) {
      const int t = warp + i * NW;
      if (t < rows) {
        kr[i].load(kb + ((size_t)t * HD + lane * DL) * 2);
        vr[i].load(vb + ((size_t)t * HD + lane * DL) * 2);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[P.slot]);
    if (FAST) {
      // partial dots of every (head, position) of this warp, then one butterfly
      float x[FAST ? V : 1];
#pragma unroll
      for (int i = 0; i < PW; ++i) {
        float kv[DL];
        kr[i].unpack(kv);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          float d = 0.f;
#pragma unroll
          for (int j = 0; j < DL; ++j) d = fmaf(qr[gg][j], kv[j], d);
          x[(gg * PW + i) % (FAST ? V : 1)] = d;
        }
      }
#pragma unroll
      for (int st = 0; st < LV; ++st) {  // halve the values held, lane bit 4 - st
        const int o = 16 >> st, half = V >> (st + 1);
        const bool upper = lane & o;
#pragma unroll
        for (int k = 0; k < half; ++k) {
          const float send = upper ? x[k] : x[k + half];
          const float keep = upper ? x[k + half] : x[k];
          x[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
#pragma unroll
      for (int o = 16 >> LV; o > 0; o >>= 1) x[0] += __shfl_xor_sync(0xffffffffu, x[0], o);
      const float sc = (warp + my_i * NW < rows) ? x[0] : -INFINITY;
      // Lazy rescaling: a head's reference max m_mine moves only when one of
      // its scores exceeds it by more than kAttnRescaleSlack, so most chunks
      // need no max, no rescale and no cross-lane sum.  The weights
      // exp(s - m_mine) stay below e^slack, and acc / l is the same ratio
      // whichever reference both carry.
      if (__any_sync(0xffffffffu, sc > m_mine + kAttnRescaleSlack)) {  // warp-uniform
        float mx = sc;
#pragma unroll
        for (int bt = 0; bt < LPW; ++bt) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1 << (SH + bt)));
        const float m_new = fmaxf(m_mine, mx);
        const float alpha = (m_mine == -INFINITY) ? 0.f : expf(m_mine - m_new);
        l_mine *= alpha;
        m_mine = m_new;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float a = __shfl_sync(0xffffffffu, alpha, (gg * PW) << SH);
#pragma unroll
          for (int j = 0; j < DL; ++j) acc[gg][j] *= a;
        }
      }
      const float pr = (sc == -INFINITY) ? 0.f : expf(sc - m_mine);
      l_mine += pr;  // this lane's (head, position) slot; the positions are summed at the segment's end
#pragma unroll
      for (int i = 0; i < PW; ++i) {
        if (warp + i * NW >= rows) break;  // warp-uniform
        float vv[DL];
        vr[i].unpack(vv);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float pi = __shfl_sync(0xffffffffu, pr, (gg * PW + i) << SH);
#pragma unroll
          for (int j = 0; j < DL; ++j) acc[gg][j] = fmaf(pi, vv[j], acc[gg][j]);
        }
      }
    }
#pragma unroll
    for (int i0 = 0; i0 < (FAST ? 0 : PW); i0 += SUB) {
      if (warp + i0 * NW >= rows) break;  // warp-uniform
      float sc[SUB][G];
#pragma unroll
      for (int i = 0; i < SUB; ++i) {
        const int t = warp + (i0 + i) * NW;
        float kv[DL];
        kr[i0 + i].unpack(kv);
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
        for (int i = 0; i < SUB; ++i) mx = fmaxf(mx, sc[i][gg]);
        const float alpha = (m[gg] == -INFINITY) ? 0.f : expf(m[gg] - mx);
        float ls = l[gg] * alpha;
#pragma unroll
        for (int j = 0; j < DL; ++j) acc[gg][j] *= alpha;
#pragma unroll
        for (int i = 0; i < SUB; ++i) {
          const int t = warp + (i0 + i) * NW;
          if (t >= rows) continue;
          const float pi = expf(sc[i][gg] - mx);
          ls += pi;
          float vv[DL];
          vr[i0 + i].unpack(vv);
#pragma unroll
          for (int j = 0; j < DL; ++j) acc[gg][j] = fmaf(pi, vv[j], acc[gg][j]);
        }
        m[gg] = mx;
        l[gg] = ls;
      }
    }
    if (++c == cph) {
      c = 0;
      ++g;
    }
    P.next(R.n);
  }
  if (tid == 0) {
    tl_mark_min(p.tl, 5);
    tl_mark_max(p.tl, 6);
  }
  if (cur_g >= 0) end_segment(cur_g);

  if (CL) {
    // ---- the cluster merges its head: CTA r finishes a slice of the G x HD outputs
    const int C = p.cluster, r = (int)cluster_rank(), gh = b / C;
    if (XG) {
      named_barrier(1, NC);  // this CTA's record (or its empty record) is written
      if (tid == 0)
        for (int c2 = 0; c2 < C; ++c2) mbar_arrive_cluster(dsmem_addr(&xg->bars[0], (uint32_t)c2));
      if (!mbar_wait_cluster(&xg->bars[0], 0, p.err)) {
        raise_error(p.err, ERR_CLUSTER_WAIT);
        ok = false;
      }
    } else {
      cluster_sync_all();  // every CTA's pushes are in this CTA's shared memory
    }
    // whole 32-element blocks per CTA (a warp finishes one block at a time)
    const int e0 = 32 * split_begin32(G * HD / 32, C, r), e1 = 32 * split_begin32(G * HD / 32, C, r + 1);
    for (int e = e0 + tid; e < e1; e += NC) {
      const int gg = e / HD, j = e - gg * HD;
      // two passes over the cluster's records in rank order: the largest
      // running max, then the rescaled sums (no per-record arrays in registers)
      float M = -INFINITY, Lsum = 0.f, o = 0.f;
      if (XG) {  // pulled from the other CTAs' records
        for (int c2 = 0; c2 < C; ++c2)
          M = fmaxf(M, dsmem_ld(dsmem_addr(crec + gg * (HD + 2), (uint32_t)c2) + 4 * HD));
        for (int c2 = 0; c2 < C; ++c2) {
          const uint32_t a = dsmem_addr(crec + gg * (HD + 2), (uint32_t)c2);
          const float mv = dsmem_ld(a + 4 * HD);
          const float w = (mv == -INFINITY) ? 0.f : expf(mv - M);
          Lsum = fmaf(dsmem_ld(a + 4 * (HD + 1)), w, Lsum);
          o = fmaf(dsmem_ld(a + 4 * j), w, o);
        }
      } else {  // pushed into this CTA's shared memory
        for (int c2 = 0; c2 < C; ++c2) M = fmaxf(M, pml[((size_t)c2 * G + gg) * 2]);
        for (int c2 = 0; c2 < C; ++c2) {
          const float mv = pml[((size_t)c2 * G + gg) * 2];
          const float w = (mv == -INFINITY) ? 0.f : expf(mv - M);
          Lsum = fmaf(pml[((size_t)c2 * G + gg) * 2 + 1], w, Lsum);
          o = fmaf(pv[(size_t)c2 * MS + (e - e0)], w, o);
        }
      }
      const size_t oi = (size_t)(gh * G + gg) * HD + j;
      if (XG) {  // into every CTA's copy of o_g
        for (int c2 = 0; c2 < C; ++c2) dsmem_st(dsmem_addr(xg->og + e, (uint32_t)c2), o / Lsum);
        continue;
      }
      p.o[oi] = o / Lsum;
      if (p.qout.codes)  // the int8 input of the o-proj, one block per warp
        q8_block_warp(o / Lsum, tid & 31, p.qout.codes + (oi & ~(size_t)31),
                      p.qout.scale + (oi >> 5), p.qout.sum + (oi >> 5));
    }
    if (XG) {
      // this CTA's pushes are done and it has read every record; o_g is complete
      // once every CTA has pushed (the records are released at the kernel's end)
      named_barrier(1, NC);
      if (tid == 0)
        for (int c2 = 0; c2 < C; ++c2) {
          mbar_arrive_cluster(dsmem_addr(&xg->bars[1], (uint32_t)c2));
          mbar_arrive_cluster(dsmem_addr(&xg->bars[2], (uint32_t)c2));
        }
      if (!mbar_wait_cluster(&xg->bars[1], 0, p.err)) {
        raise_error(p.err, ERR_CLUSTER_WAIT);
        ok = false;
      }
      return ok;
    }
    return ok;  // nothing is read from another CTA after the barrier
  }

  // ---- heads split over CTAs: the last CTA to finish merges them --------------
  // (tickets are taken after this CTA's whole loop, so merging never stalls it;
  // the split arithmetic is 32-bit: units * grid stays far below 2^31)
  int* mbase = reinterpret_cast<int*>(work + AL.merge_off());  // [2][kMaxSplits]
  int* todo = mbase + 2 * kMaxSplits;                                         // [2]: head, splits
  const int U32 = U;
  auto part_begin = [&](int c) { return split_begin32(U32, nb, c); };
  if (tid < 2) {
    // thread i takes the ticket of this CTA's i-th split head (both in flight at once)
    const int g = split_heads[tid];
    int head = -1;
    if (g >= 0) {
      const int c_lo = split_owner32(U32, nb, g * cph), c_hi = split_owner32(U32, nb, (g + 1) * cph - 1);
      int expected = 0;
      for (int c = c_lo; c <= c_hi; ++c) expected += part_begin(c + 1) > part_begin(c);
      // release this CTA's record, acquire the others'
      if (atomic_add_acq_rel(&p.counters[g], 1) == expected - 1) head = g;
    }
    todo[tid] = head;
  }
  named_barrier(1, NC);
  // record offset of every split of the heads to merge
  for (int t = tid; t < 2 * kMaxSplits; t += NC) {
    const int i = t / kMaxSplits, sp = t - i * kMaxSplits, g = todo[i];
    int off = -1;
    if (g >= 0) {
      const int h0 = g * cph, c_lo = split_owner32(U32, nb, h0);
      const int c_hi = split_owner32(U32, nb, h0 + cph - 1);
      if (sp == 0 && c_hi - c_lo + 1 > kMaxSplits) raise_error(p.err, ERR_SPLITS);
      const int c = c_lo + sp;
      if (c <= c_hi && TLD_IN_BOUNDS(c >= 0 && c < nb && g < p.nkv, p.err)) {
        const int cs = part_begin(c);
        if (part_begin(c + 1) > cs) off = ((c * 2 + (cs >= h0 ? 0 : 1)) * G) * (HD + 4);
      }
    }
    mbase[t] = off;
  }
  named_barrier(1, NC);
  // both heads at once; one round trip: each output loads every split's
  // (m, l, acc) together, then combines them in split order
  for (int t = tid; t < 2 * G * HD; t += NC) {
    const int i = t / (G * HD), e = t - i * G * HD;
    const int g = todo[i];
    if (g < 0) continue;
    const int gg = e / HD, j = e - gg * HD;
    const int* mb = mbase + i * kMaxSplits;
    // two passes over the head's split records in split order: the largest
    // running max, then the rescaled sums (no per-split arrays in registers)
    float M = -INFINITY;
    for (int sp = 0; sp < kMaxSplits; ++sp) {
      const int off = mb[sp];
      if (off >= 0) M = fmaxf(M, __ldcg(p.part + off + gg * (HD + 4) + HD));
    }
    float Lsum = 0.f, o = 0.f;
    for (int sp = 0; sp < kMaxSplits; ++sp) {
      const int off = mb[sp];
      if (off < 0) continue;
      const float* rec = p.part + off + gg * (HD + 4);
      const float mv = __ldcg(rec + HD);
      const float w = (mv == -INFINITY) ? 0.f : expf(mv - M);
      Lsum = fmaf(__ldcg(rec + HD + 1), w, Lsum);
      o = fmaf(__ldcg(rec + j), w, o);
    }
    const size_t oi = (size_t)(g * G + gg) * HD + j;
    p.o[oi] = o / Lsum;
    if (p.qout.codes)  // the int8 input of the o-proj, one block per warp
      q8_block_warp(o / Lsum, tid & 31, p.qout.codes + (oi & ~(size_t)31), p.qout.scale + (oi >> 5),
                    p.qout.sum + (oi >> 5));
  }
  if (tid < 2 && todo[tid] >= 0) p.counters[todo[tid]] = 0;
  named_barrier(1, NC);
  return ok;
}

// ---- o-projection by KV-head group (the attention + head-projection kernel) ----
// Work area after the attention's: the group's merged output o_g, its int8
// codes (q4), the scratch of the final sum over groups, the three exchange
// mbarriers and the last-arrival flag.
struct HeadProjLayout {
  int hd, G, quads, nh;  // quads: row quads per CTA at most; nh: 16-group chunks of the sum
  bool q4;
  __host__ __device__ size_t attn_bytes() const { return (AttnLayout{hd, G, kConsumerWarps}.total() + 15) & ~(size_t)15; }
  __host__ __device__ size_t og_off() const { return attn_bytes(); }
  __host__ __device__ size_t qx_off() const { return og_off() + 4 * (size_t)G * hd; }
  __host__ __device__ size_t dx_off() const { return qx_off() + (q4 ? (size_t)G * hd : 0); }
  __host__ __device__ size_t sx_off() const { return dx_off() + (q4 ? 4 * (size_t)G * hd / 32 : 0); }
  __host__ __device__ size_t red_off() const { return (sx_off() + (q4 ? 4 * (size_t)G * hd / 32 : 0) + 15) & ~(size_t)15; }
  __host__ __device__ size_t bar_off() const { return red_off() + 16 * (size_t)quads * nh; }
  __host__ __device__ size_t total() const { return bar_off() + 3 * 8 + 8; }
};

// Producer: rows [rb0, rb1) of a group's tiled matrix, as many whole row
// blocks per stage as a ring slot holds.
__device__ __forceinline__ void rows_produce(const uint8_t* w, const TileGeom& geo, int rb0, int rb1,
                                             const Ring& R, RingPos& P, uint64_t pol, int* err) {
  const int rps = (int)(R.slot_bytes / geo.rb_bytes);
  if (!TLD_IN_BOUNDS(rps >= 1 && (geo.rb_bytes & 15) == 0, err)) return;
  for (int rb = rb0; rb < rb1; rb += rps) {
    const int n = rb1 - rb < rps ? rb1 - rb : rps;
    if (!ring_reserve(R, P, err)) return;
    const uint32_t bytes = (uint32_t)(n * geo.rb_bytes);
    mbar_arrive_expect_tx(&R.full[P.slot], bytes);
    bulk_g2s_split(R.slot(P.slot), w + (int64_t)rb * geo.rb_bytes, bytes, &R.full[P.slot], pol,
                   geo.copies);
    P.next(R.n);
  }
}

// Consumers: x (fp32 [K], or its int8 codes qx / dx / sx for q4 weights) times
// rows [rb0, rb1) of the tiled matrix streamed by rows_produce.  A warp takes
// whole row blocks (every k-tile of them), so each row is finished inside one
// warp: emit(row, value) is called by lane 8r of the warp for row r of the
// block.  dots (q4, optional): the integer block dots, row-major with ld
// blocks per row.  Returns false if a wait ran out.
template <bool Q4, class Emit>
__device__ __forceinline__ bool rows_main(const TileGeom& geo, const float* x, const uint8_t* qx,
                                          const float* dx, const int* sx, const Ring& R, RingPos& P,
                                          int rb0, int rb1, int tid, int* err, int32_t* dots,
                                          int dots_ld, Emit&& emit) {
  const int warp = tid >> 5, lane = tid & 31;
  const int rps = (int)(R.slot_bytes / geo.rb_bytes);
  bool ok = rps >= 1;
  for (int rbs = rb0; rbs < rb1 && rps >= 1; rbs += rps) {
    const int n = rb1 - rbs < rps ? rb1 - rbs : rps;
    if (ok && !mbar_wait(&R.full[P.slot], P.phase, err)) {
      raise_error(err, ERR_FULL_WAIT);
      ok = false;
    }
    const uint8_t* st = R.slot(P.slot);
    for (int i = warp; ok && i < n; i += kConsumerWarps) {
      const int rb = rbs + i;
      float acc[kTileR] = {0.f, 0.f, 0.f, 0.f};
      for (int kt = 0; kt < geo.ktiles; ++kt) {
        const int kw = (kt == geo.ktiles - 1) ? geo.kw_last : geo.tile_k;
        const uint8_t* tp = st + (int64_t)i * geo.rb_bytes + (int64_t)kt * geo.tile_bytes;
        if (Q4) {
          if (lane * 32 >= kw) continue;
          const int blk = kt * (kTileKQ4 / 32) + lane;
          const uint4 x0 = *reinterpret_cast<const uint4*>(qx + blk * 32);
          const uint4 x1 = *reinterpret_cast<const uint4*>(qx + blk * 32 + 16);
          const uint2 sc = *reinterpret_cast<const uint2*>(tp + (size_t)kTileR * (kw / 2) + lane * 8);
          const uint32_t sc2[2] = {sc.x, sc.y};
#pragma unroll
          for (int r = 0; r < kTileR; ++r) {
            const uint4 wv = *reinterpret_cast<const uint4*>(tp + (size_t)r * (kw / 2) + lane * 16);
            const int idot = q4_block_dot(wv, x0, x1, sx[blk]);
            const uint16_t hb = (uint16_t)(r & 1 ? sc2[r >> 1] >> 16 : sc2[r >> 1] & 0xffff);
            acc[r] = fmaf(__half2float(__ushort_as_half(hb)) * dx[blk], (float)idot, acc[r]);
            if (dots) dots[(size_t)(rb * kTileR + r) * dots_ld + blk] = idot;
          }
        } else {
          const int c = lane * 8;
          if (c >= kw) continue;
          const float4 xa = *reinterpret_cast<const float4*>(x + kt * kTileK + c);
          const float4 xb = *reinterpret_cast<const float4*>(x + kt * kTileK + c + 4);
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
      const float v = warp_reduce4(acc, lane);
      if ((lane & 7) == 0) emit(rb * kTileR + (lane >> 3), v);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[P.slot]);
    P.next(R.n);
  }
  return ok;
}

// The last of the nkv CTAs that cover rows [r0, r1) (one per KV-head group)
// adds their partial projections in group order to the residual:
// out = resid + sum_g part[g].  Sixteen groups' float4 loads in flight per
// thread; the chunks of sixteen groups are added in chunk order.
__device__ __forceinline__ void headproj_sum(const float* part, int nkv, int H, const float* resid,
                                             float* out, float* tap, int r0, int r1, float4* red,
                                             int tid, int NC) {
  const int quads = (r1 - r0) / 4, nh = (nkv + 15) / 16;
  for (int t = tid; t < quads * nh; t += NC) {
    const int q = t % quads, h = t / quads;
    const int row = r0 + 4 * q;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (16 * h + i < nkv)
        v[i] = __ldcg(reinterpret_cast<const float4*>(part + (size_t)(16 * h + i) * H + row));
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (16 * h + i < nkv) {
        a.x += v[i].x;
        a.y += v[i].y;
        a.z += v[i].z;
        a.w += v[i].w;
      }
    red[h * quads + q] = a;
  }
  named_barrier(1, NC);
  for (int q = tid; q < quads; q += NC) {
    const int row = r0 + 4 * q;
    float4 a = red[q];
    for (int h = 1; h < nh; ++h) {
      const float4 b = red[h * quads + q];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    const float4 x = __ldcg(reinterpret_cast<const float4*>(resid + row));
    const float4 y = make_float4(x.x + a.x, x.y + a.y, x.z + a.z, x.w + a.w);
    *reinterpret_cast<float4*>(out + row) = y;
    if (tap) *reinterpret_cast<float4*>(tap + row) = y;
  }
}

}  // namespace tld
