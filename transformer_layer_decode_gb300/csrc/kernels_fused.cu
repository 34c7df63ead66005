// Fused decode-layer kernels for sm_103a.
//
// Five kernels per layer (the fusions of "RDNA4 Decode Kernel Fusion:
// Pipeline Barriers, Not Launches, Are the Win", FAQ and section "Fusion
// removes the barrier by removing the write"):
//   K1 gemv<PRO_NORM,  EPI_QKV>    RMSNorm*w, [Wq;Wk;Wv] GEMV, RoPE on q and k
//                                  and the k/v append in the epilogue
//   K2 attn_decode                 GQA split-KV attention; a head split over
//                                  CTAs is merged by the last one to finish
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
// thread.  Eight consumer warps each take two 4-row x 256-column tiles per
// stage, copy them to registers, hand the stage back, and accumulate against
// the input vector held in shared memory in fp32.  Because CTAs own whole rows,
// no partial sums cross CTAs.  Weights do not depend on the previous kernel:
// the producer starts streaming at launch, before griddepcontrol.wait.
#include "common.cuh"
#include "kernels.h"

namespace tld {

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// ---- shared memory layout of the GEMV kernel -------------------------------
// ring of stages | mbarriers | x (fp32, K) | [q4: int8 x (K), block scales,
// block sums] | per-warp row-block partials | warp sums
struct GemvSmem {
  int K, nstages, max_rb_local, stage_bytes;
  bool q4;
  __host__ __device__ size_t bars_off() const { return (size_t)nstages * stage_bytes; }
  __host__ __device__ size_t xs_off() const { return bars_off() + 16 * (size_t)nstages; }
  __host__ __device__ size_t qx_off() const { return xs_off() + 4 * (size_t)((K + 3) & ~3); }
  __host__ __device__ size_t dx_off() const { return qx_off() + (q4 ? (size_t)K : 0); }
  __host__ __device__ size_t sx_off() const { return dx_off() + (q4 ? 4 * (size_t)(K / 32) : 0); }
  __host__ __device__ size_t part_off() const {
    return sx_off() + (q4 ? 4 * (size_t)(K / 32) : 0);
  }
  __host__ __device__ size_t red_off() const {
    return part_off() + 4 * (size_t)max_rb_local * kConsumerWarps * kTileR;
  }
  __host__ __device__ size_t total() const { return red_off() + 4 * 32; }  // warp sums + abort mark
};

size_t gemv_smem_bytes(int K, bool q4, int nstages, int max_rb_local) {
  return GemvSmem{K, nstages, max_rb_local, q4 ? kStageBytesQ4 : kStageBytes, q4}.total();
}

// Epilogue of one finished row block (kTileR tiled rows, values v).
template <int EPI>
__device__ __forceinline__ void gemv_epilogue(const GemvParams& p, int rb, const float v[kTileR]) {
  const int R0 = rb * kTileR;
  if (EPI == EPI_QKV) {
    const int hd = p.hd, half = hd / 2;
    const int qrows = p.nq * hd, krows = p.nkv * hd;
    const int pos = *p.pos;
    if (R0 < qrows + krows) {
      // rows (2i, 2i+1) of a head hold dims i and i + hd/2: rotate the pair
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
      for (int r = 0; r < kTileR; ++r) row[j + r] = f32_to_bf16_bits(v[r]);
    }
  } else if (EPI == EPI_RESID) {
#pragma unroll
    for (int r = 0; r < kTileR; ++r) {
      const float y = p.resid[R0 + r] + v[r];
      p.out[R0 + r] = y;
      if (p.tap) p.tap[R0 + r] = y;
    }
  } else {  // EPI_SWIGLU: tiled rows alternate gate and up of the same output
    const int j = R0 / 2;
#pragma unroll
    for (int pr = 0; pr < kTileR / 2; ++pr) p.a_out[j + pr] = silu_f(v[2 * pr]) * v[2 * pr + 1];
  }
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
__device__ void quantize_blocks(const float* xs, int K, uint8_t* qx, float* dx, int* sx,
                                int8_t* qtap, float* qstap, int tid, int NC) {
  const int lane = tid & 31, sub = lane & 7, warp = tid >> 5;
  const int nblk = K / 32;
  // Four blocks per warp per round; the round count is the same for all lanes
  // of a warp (the shuffles below name the whole warp).
  for (int base = warp * 4; base < nblk; base += (NC >> 5) * 4) {
    const int blk = base + (lane >> 3);
    const bool live = blk < nblk;
    const int e = blk * 32 + sub * 4;
    const float4 z = live ? *reinterpret_cast<const float4*>(xs + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    float amax = fmaxf(fmaxf(fabsf(z.x), fabsf(z.y)), fmaxf(fabsf(z.z), fabsf(z.w)));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    int q[4];
    const float zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int v = 0;
      if (d != 0.0f) {
        v = __float2int_rn(__fdiv_rn(zz[i], d));
        v = v > 127 ? 127 : (v < -127 ? -127 : v);
      }
      q[i] = v;
    }
    int sum = q[0] + q[1] + q[2] + q[3];
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (!live) continue;
    // elements e..e+3 = 8g + 4h + {0,1,2,3}: evens go to bytes 8g+2h, 8g+2h+1,
    // odds to bytes 8g+4+2h, 8g+4+2h+1
    const int g8 = e & ~7, h = (e >> 2) & 1;
    *reinterpret_cast<uint16_t*>(qx + g8 + 2 * h) = (uint16_t)((q[0] & 0xff) | ((q[2] & 0xff) << 8));
    *reinterpret_cast<uint16_t*>(qx + g8 + 4 + 2 * h) =
        (uint16_t)((q[1] & 0xff) | ((q[3] & 0xff) << 8));
    if (sub == 0) {
      dx[blk] = d;
      sx[blk] = sum;
    }
    if (qtap) {
#pragma unroll
      for (int i = 0; i < 4; ++i) qtap[e + i] = (int8_t)q[i];
      if (sub == 0) qstap[blk] = d;
    }
  }
}

// Integer dot of one 32-block: packed nibbles (q + 8) against the arranged
// int8 activations, minus 8 * (sum of the activations).
__device__ __forceinline__ int q4_block_dot(const uint4 w, const uint4 x0, const uint4 x1, int sx) {
  constexpr uint32_t M = 0x0F0F0F0Fu;
  int d = 0;
  d = __dp4a((int)(w.x & M), (int)x0.x, d);
  d = __dp4a((int)((w.x >> 4) & M), (int)x0.y, d);
  d = __dp4a((int)(w.y & M), (int)x0.z, d);
  d = __dp4a((int)((w.y >> 4) & M), (int)x0.w, d);
  d = __dp4a((int)(w.z & M), (int)x1.x, d);
  d = __dp4a((int)((w.z >> 4) & M), (int)x1.y, d);
  d = __dp4a((int)(w.w & M), (int)x1.z, d);
  d = __dp4a((int)((w.w >> 4) & M), (int)x1.w, d);
  return d - 8 * sx;
}

template <int PRO, int EPI, bool Q4>
__global__ void __launch_bounds__(kThreads, 1) gemv_fused(const GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const TileGeom& geo = p.geo;
  const int K = geo.K;
  const GemvSmem L{K, p.nstages, p.max_rb_local, geo.stage_bytes, Q4};
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars_off());
  uint64_t* empty = full + p.nstages;
  float* xs = reinterpret_cast<float*>(smem + L.xs_off());
  uint8_t* qx = smem + L.qx_off();
  float* dxs = reinterpret_cast<float*>(smem + L.dx_off());
  int* sxs = reinterpret_cast<int*>(smem + L.sx_off());
  float* part_s = reinterpret_cast<float*>(smem + L.part_off());
  float* red = reinterpret_cast<float*>(smem + L.red_off());

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  if (tid == 0) tl_mark_min(p.tl, 0);
  // whole row blocks [rb0, rb1) of this CTA = tiles [rb0 * ktiles, rb1 * ktiles)
  const int rb0 = (int)split_begin(p.n_rb, nb, b), rb1 = (int)split_begin(p.n_rb, nb, b + 1);
  const int nrb = rb1 - rb0;
  const int nloc = nrb * geo.ktiles;
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
      TileCursor cur{rb0, 0};
      const int64_t end_off = (int64_t)rb1 * geo.rb_bytes;
      const uint64_t pol_stream = policy_evict_first();
      int slot = 0, phase = 0;
      for (int s = 0; s < nst; ++s) {
        if (s >= p.nstages && !mbar_wait(&empty[slot], phase ^ 1)) {
          raise_error(p.err, ERR_EMPTY_WAIT);
          break;
        }
        const int64_t oa = cur.offset(geo);
        cur.advance(kStageTiles, geo.ktiles);
        const int64_t ob = (s == nst - 1) ? end_off : cur.offset(geo);
        const uint32_t bytes = (uint32_t)(ob - oa);
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s_hint(stages + (size_t)slot * geo.stage_bytes, p.w + oa, bytes, &full[slot],
                      pol_stream);
        if (++slot == p.nstages) {
          slot = 0;
          phase ^= 1;
        }
      }
    }
    return;
  }

  // ---- consumers -------------------------------------------------------------
  constexpr int NC = kConsumerWarps * 32;
  const int K4 = K / 4;
  // Before the wait: the RMSNorm weights (static) go to xs as fp32.
  if (PRO == PRO_NORM) {
    const uint2* w4 = reinterpret_cast<const uint2*>(p.norm_w);
    for (int k4 = tid; k4 < K4; k4 += NC) {
      const uint2 wb = w4[k4];
      reinterpret_cast<float4*>(xs)[k4] =
          make_float4(bf16lo(wb.x), bf16hi(wb.x), bf16lo(wb.y), bf16hi(wb.y));
    }
  }
  for (int i = tid; i < p.max_rb_local * kConsumerWarps * kTileR; i += NC) part_s[i] = 0.f;
  if (tid == 0) red[kConsumerWarps] = 0.f;

  pdl_wait();  // the input vector comes from the previous kernel
  if (tid == 0) {
    tl_mark_min(p.tl, 2);
    tl_mark_max(p.tl, 3);
  }
  // Let the next kernel launch (and start its weight stream) now.  Triggering
  // only after this CTA's own wait keeps at most two kernels in flight and means
  // everything before the previous kernel is complete when the next one starts.
  pdl_trigger();

  {
    const float4* x4 = reinterpret_cast<const float4*>(p.x);
    float ss = 0.f;
    constexpr int PB = 4;  // loads in flight per thread
    for (int base = tid; base < K4; base += NC * PB) {
      float4 v[PB];
#pragma unroll
      for (int u = 0; u < PB; ++u)
        if (base + u * NC < K4) v[u] = x4[base + u * NC];
#pragma unroll
      for (int u = 0; u < PB; ++u) {
        const int k4 = base + u * NC;
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
      if (lane == 0) red[warp] = ss;
    }
  }
  if (p.x_copy && b == 0) {
    for (int k = tid; k < K; k += NC) p.x_copy[k] = p.x[k];
  }
  if (p.pos_advance && b == 0 && tid == 0) atomicAdd(p.pos_advance, 1);
  named_barrier(1, NC);

  // RMSNorm is a per-vector scale 1/sqrt(mean(x^2)+eps).  bf16 weights: the
  // projection runs on x*w and the scale multiplies the finished rows.  q4
  // weights: the normalised vector itself is quantised, so it is scaled first.
  float rnorm = 1.f;
  if (PRO == PRO_NORM) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += red[w];
    rnorm = 1.0f / sqrtf(tot / (float)K + p.eps);
  }
  if (Q4) {
    if (PRO == PRO_NORM) {
      for (int k4 = tid; k4 < K4; k4 += NC) {
        float4 v = reinterpret_cast<float4*>(xs)[k4];
        v.x *= rnorm;
        v.y *= rnorm;
        v.z *= rnorm;
        v.w *= rnorm;
        reinterpret_cast<float4*>(xs)[k4] = v;
      }
      named_barrier(1, NC);
      rnorm = 1.f;
    }
    quantize_blocks(xs, K, qx, dxs, sxs, b == 0 ? p.qtap : nullptr, p.qstap, tid, NC);
    named_barrier(1, NC);
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
  int slot = 0, phase = 0;
  for (int s = 0; s < nst; ++s) {
    // After a timed-out wait the warp stops waiting but keeps the same control
    // flow, so that every named barrier below is still reached by all warps.
    if (ok && !mbar_wait(&full[slot], phase)) {
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
      if (li < nloc && c < kw) {
        const uint8_t* tp = stages + (size_t)slot * geo.stage_bytes + (my[j].offset(geo) - st_off);
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
    if (lane == 0) mbar_arrive(&empty[slot]);
#pragma unroll
    for (int j = 0; j < kTilesPerWarp; ++j) {
      const int li = s * kStageTiles + warp + j * kConsumerWarps;
      if (li >= nloc) continue;
      const int rb = my[j].rb, kt = my[j].kt;
      if (rb != cur_rb) {
        if (cur_rb >= 0) {
          const float v = warp_reduce4(acc, lane);
          if ((lane & 7) == 0)
            part_s[((cur_rb - rb0) * kConsumerWarps + warp) * kTileR + (lane >> 3)] = v;
        }
        cur_rb = rb;
#pragma unroll
        for (int r = 0; r < kTileR; ++r) acc[r] = 0.f;
      }
      const int kw = (kt == geo.ktiles - 1) ? geo.kw_last : geo.tile_k;
      if (c >= kw) continue;
      if (Q4) {
        const int blk = kt * (kTileKQ4 / 32) + lane;
        const uint4 x0 = *reinterpret_cast<const uint4*>(qx + blk * 32);
        const uint4 x1 = *reinterpret_cast<const uint4*>(qx + blk * 32 + 16);
        const float dxb = dxs[blk];
        const int sxb = sxs[blk];
        const uint32_t sc2[2] = {scl[j].x, scl[j].y};
#pragma unroll
        for (int r = 0; r < kTileR; ++r) {
          const int idot = q4_block_dot(wv[j][r], x0, x1, sxb);
          const uint16_t hb = (uint16_t)(r & 1 ? sc2[r >> 1] >> 16 : sc2[r >> 1] & 0xffff);
          const float sw = __half2float(__ushort_as_half(hb));
          acc[r] = fmaf(sw * dxb, (float)idot, acc[r]);
          if (p.dots) p.dots[(size_t)(rb * kTileR + r) * (K / 32) + blk] = idot;
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
    if (++slot == p.nstages) {
      slot = 0;
      phase ^= 1;
    }
  }
  if (cur_rb >= 0) {
    const float v = warp_reduce4(acc, lane);
    if ((lane & 7) == 0)
      part_s[((cur_rb - rb0) * kConsumerWarps + warp) * kTileR + (lane >> 3)] = v;
  }
  if (!ok && lane == 0) red[kConsumerWarps] = 1.f;  // abort mark
  named_barrier(1, NC);
  if (tid == 0) {
    tl_mark_min(p.tl, 5);
    tl_mark_max(p.tl, 6);
  }
  if (red[kConsumerWarps] != 0.f) {
    // Drain: wait (bounded) for the last copy into every slot, then leave.
    if (tid == 0)
      for (int s = 0; s < nst && s < p.nstages; ++s) {
        const int last = s + ((nst - 1 - s) / p.nstages) * p.nstages;
        if (!mbar_wait(&full[s], (last / p.nstages) & 1)) raise_error(p.err, ERR_DRAIN);
      }
    return;
  }

  // ---- finish this CTA's row blocks (sum over warps in warp order) ------------
  for (int j = tid; j < nrb; j += NC) {
    float v[kTileR];
#pragma unroll
    for (int r = 0; r < kTileR; ++r) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) sum += part_s[(j * kConsumerWarps + w) * kTileR + r];
      v[r] = sum * rnorm;
    }
    gemv_epilogue<EPI>(p, rb0 + j, v);
  }
  if (p.tl) {
    named_barrier(1, NC);
    if (tid == 0) {
      tl_mark_max(p.tl, 1);
      tl_mark_min(p.tl, 7);
    }
  }
}

// ---- attention ---------------------------------------------------------------
// One unit = one chunk of CH cached positions of one KV head (K and V rows,
// 8 KB each).  The grid splits the units of all KV heads evenly; every CTA
// serves all G query heads of the KV heads it touches, so each K/V byte is
// read once.  Within a CTA the 8 consumer warps take interleaved positions of
// each chunk and keep a running (max, sum, acc) per query head; warps are
// merged at the end of each head segment, and a head cut between CTAs is
// merged by the o-projection kernel, in CTA order.

struct AttnSmem {
  int hd, G, nstages;
  __host__ __device__ size_t bars_off() const { return (size_t)nstages * kAttnStageBytes; }
  __host__ __device__ size_t ws_off() const { return bars_off() + 16 * (size_t)nstages; }
  __host__ __device__ size_t merge_off() const {
    return ws_off() + 4 * (size_t)kConsumerWarps * G * (hd + 2);
  }
  // merge scratch: the record offset per split, then the heads to merge
  __host__ __device__ size_t total() const { return merge_off() + 4 * (size_t)kMaxSplits + 16; }
};

size_t attn_smem_bytes(int hd, int G, int nstages) { return AttnSmem{hd, G, nstages}.total(); }

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

template <int HD, int G>
__global__ void __launch_bounds__(kThreads, 1) attn_decode(const AttnParams p) {
  constexpr int CH = kAttnStageBytes / 2 / (HD * 2);  // positions per chunk (16 KB of K)
  constexpr int PW = CH / kConsumerWarps;  // positions per warp per chunk
  constexpr int SUB = 4;                   // positions per online-softmax update
  constexpr int DL = HD / 32;          // dims per lane
  constexpr int NC = kConsumerWarps * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  const AttnSmem L{HD, G, p.nstages};
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars_off());
  uint64_t* empty = full + p.nstages;
  float* ws = reinterpret_cast<float*>(smem + L.ws_off());    // [warp][G][HD+2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, b = blockIdx.x;
  if (tid == 0) tl_mark_min(p.tl, 0);
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
      int g = (int)(u0 / cph), c = (int)(u0 - (int64_t)g * cph);
      const uint64_t pol_stream = policy_evict_first();
      int slot = 0, phase = 0;
      for (int s = 0; s < nu; ++s) {
        if (s >= p.nstages && !mbar_wait(&empty[slot], phase ^ 1)) {
          raise_error(p.err, ERR_EMPTY_WAIT);
          break;
        }
        const int rows = min(CH, n - c * CH);
        if (c == cph - 1 && !waited) {  // this chunk holds the row appended by K1
          pdl_wait();
          waited = true;
        }
        const size_t off = ((size_t)g * p.max_ctx + (size_t)c * CH) * HD;
        const uint32_t bytes = (uint32_t)rows * HD * 2;
        mbar_arrive_expect_tx(&full[slot], 2 * bytes);
        uint8_t* dst = stages + (size_t)slot * kAttnStageBytes;
        bulk_g2s_hint(dst, p.kc + off, bytes, &full[slot], pol_stream);
        bulk_g2s_hint(dst + kAttnStageBytes / 2, p.vc + off, bytes, &full[slot], pol_stream);
        if (++c == cph) {
          c = 0;
          ++g;
        }
        if (++slot == p.nstages) {
          slot = 0;
          phase ^= 1;
        }
      }
    }
    return;
  }

  pdl_wait();  // q comes from K1
  pdl_trigger();
  if (tid == 0) {
    tl_mark_min(p.tl, 2);
    tl_mark_max(p.tl, 3);
  }
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
  // Ends the segment of KV head g: merge the warps' states; a head this CTA
  // covered whole is normalised into o, a split head leaves a partial record
  // (acc, m, l), merged after the loop by the last CTA of the head to finish.
  int split_heads[2] = {-1, -1};
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
    const int64_t h0 = (int64_t)g * cph, h1 = h0 + cph;
    const bool whole = h0 >= u0 && h1 <= u1;
    if (!whole) split_heads[seg_idx == 0 ? 0 : 1] = g;
    float* rec = p.part + ((size_t)b * 2 + (seg_idx == 0 ? 0 : 1)) * G * (HD + 4);
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
      if (whole) {
        p.o[(size_t)(g * G + gg) * HD + j] = A / Ls;
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
  bool ok = true;
  int g = (int)(u0 / cph), c = (int)(u0 - (int64_t)g * cph);
  int slot = 0, phase = 0;
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
        for (int j = 0; j < DL; ++j) qr[gg][j] = p.q[(size_t)(g * G + gg) * HD + lane * DL + j] * p.scale;
    }
    if (ok && !mbar_wait(&full[slot], phase)) {
      raise_error(p.err, ERR_FULL_WAIT);
      ok = false;  // keep the control flow (segment barriers) uniform
    }
    if (s == 0 && tid == 0) tl_mark_max(p.tl, 4);
    const int rows = min(CH, n - c * CH);
    const uint8_t* kb = stages + (size_t)slot * kAttnStageBytes;
    const uint8_t* vb = kb + kAttnStageBytes / 2;
    // This warp's K and V row slices into registers, then the slot goes back.
    RowSlice<DL> kr[PW], vr[PW];
#pragma unroll
    for (int i = 0; i < PW; ++i) {
      const int t = warp + i * kConsumerWarps;
      if (t < rows) {
        kr[i].load(kb + ((size_t)t * HD + lane * DL) * 2);
        vr[i].load(vb + ((size_t)t * HD + lane * DL) * 2);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
#pragma unroll
    for (int i0 = 0; i0 < PW; i0 += SUB) {
      if (warp + i0 * kConsumerWarps >= rows) break;  // warp-uniform
      float sc[SUB][G];
#pragma unroll
      for (int i = 0; i < SUB; ++i) {
        const int t = warp + (i0 + i) * kConsumerWarps;
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
          const int t = warp + (i0 + i) * kConsumerWarps;
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
    if (++slot == p.nstages) {
      slot = 0;
      phase ^= 1;
    }
  }
  if (tid == 0) {
    tl_mark_min(p.tl, 5);
    tl_mark_max(p.tl, 6);
  }
  if (cur_g >= 0) end_segment(cur_g);

  // ---- heads split over CTAs: the last CTA to finish merges them --------------
  // (tickets are taken after this CTA's whole loop, so merging never stalls it;
  // the split arithmetic is 32-bit: units * grid stays far below 2^31)
  int* mbase = reinterpret_cast<int*>(smem + L.merge_off());  // [kMaxSplits] record offset
  int* todo = mbase + kMaxSplits;                              // [2]
  const int U32 = (int)U;
  auto part_begin = [&](int c) { return split_begin32(U32, nb, c); };
  if (tid == 0) {
    int prev[2] = {0, 0}, expected[2] = {0, 0};
    for (int i = 0; i < 2; ++i) {
      const int g = split_heads[i];
      if (g < 0) continue;
      const int c_lo = split_owner32(U32, nb, g * cph), c_hi = split_owner32(U32, nb, (g + 1) * cph - 1);
      for (int c = c_lo; c <= c_hi; ++c) expected[i] += part_begin(c + 1) > part_begin(c);
      // release this CTA's record, acquire the others'
      prev[i] = atomic_add_acq_rel(&p.counters[g], 1);
    }
    for (int i = 0; i < 2; ++i)
      todo[i] = (split_heads[i] >= 0 && prev[i] == expected[i] - 1) ? split_heads[i] : -1;
  }
  named_barrier(1, NC);
  for (int i = 0; i < 2; ++i) {
    const int g = todo[i];
    if (g < 0) continue;
    const int h0 = g * cph;
    const int c_lo = split_owner32(U32, nb, h0), c_hi = split_owner32(U32, nb, h0 + cph - 1);
    const int S = min(c_hi - c_lo + 1, kMaxSplits);
    if (tid == 0 && c_hi - c_lo + 1 > kMaxSplits) raise_error(p.err, ERR_SPLITS);
    // record offset of every split
    for (int sp = tid; sp < S; sp += NC) {
      const int c = c_lo + sp, cs = part_begin(c);
      mbase[sp] = part_begin(c + 1) > cs ? ((c * 2 + (cs >= h0 ? 0 : 1)) * G) * (HD + 4) : -1;
    }
    named_barrier(1, NC);
    // one round trip: each output loads every split's (m, l, acc) at once
    for (int t = tid; t < G * HD; t += NC) {
      const int gg = t / HD, j = t - gg * HD;
      float mv[kMaxSplits], lv[kMaxSplits], av[kMaxSplits];
      float M = -INFINITY;
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp) {
        mv[sp] = -INFINITY;
        lv[sp] = 0.f;
        av[sp] = 0.f;
        if (sp < S && mbase[sp] >= 0) {
          const float* rec = p.part + mbase[sp] + gg * (HD + 4);
          mv[sp] = __ldcg(rec + HD);
          lv[sp] = __ldcg(rec + HD + 1);
          av[sp] = __ldcg(rec + j);
        }
      }
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp) M = fmaxf(M, mv[sp]);
      float Lsum = 0.f, o = 0.f;
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp) {
        const float e = (mv[sp] == -INFINITY) ? 0.f : expf(mv[sp] - M);
        Lsum = fmaf(lv[sp], e, Lsum);
        o = fmaf(av[sp], e, o);
      }
      p.o[(size_t)(g * G + gg) * HD + j] = o / Lsum;
    }
    if (tid == 0) p.counters[g] = 0;
    named_barrier(1, NC);
  }
  if (p.tl) {
    named_barrier(1, NC);
    if (tid == 0) {
      tl_mark_max(p.tl, 1);
      tl_mark_min(p.tl, 7);
    }
  }
  if (!ok) {
    for (int s = 0; s < nu && s < p.nstages; ++s) {
      const int last = s + ((nu - 1 - s) / p.nstages) * p.nstages;
      if (!mbar_wait(&full[s], (last / p.nstages) & 1)) raise_error(p.err, ERR_DRAIN);
    }
  }
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
  for (int hd : {64, 128})
    for (int G : {1, 2, 4, 8}) {
      cudaError_t e = cudaFuncSetAttribute(attn_kernel_ptr(hd, G),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

static cudaError_t launch_pdl(const void* fn, void** args, int grid, size_t smem, cudaStream_t s,
                              bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
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
  const void* fn = attn_kernel_ptr(hd, G);
  if (!fn) return cudaErrorInvalidValue;
  AttnParams copy = p;
  void* args[] = {&copy};
  return launch_pdl(fn, args, grid, smem, s, pdl);
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

cudaError_t launch_repack_q4(const uint8_t* nibbles, const uint16_t* scales, int rows, int K,
                             uint8_t* dst_tiled, int dst_row0, int kind, int hd, cudaStream_t s) {
  const int grid = rows < 4096 ? rows : 4096;
  repack_q4_kernel<<<grid, 256, 0, s>>>(nibbles, scales, rows, K, dst_tiled, dst_row0, kind, hd);
  return cudaGetLastError();
}

}  // namespace tld
