// The unfused decode layer: one kernel per op, intermediates round-tripping
// through global memory.  It is the ablation the fused plan is measured
// against and the per-op chain it must agree with ("Backend-Specific Kernel
// Fusion", section "A practical engineering example": keep the known-correct
// route, switchable; "Kernel fusion and block bridging", section "What it
// keeps": per-op kernels stay the reference).  The ops and their order are the
// layer chain of "RDNA4 Decode Kernel Fusion: Pipeline Barriers, Not Launches,
// Are the Win", section "Decode is where the bubble has nowhere to go".
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace tld {
namespace unf {

// RMSNorm scale: n = x / sqrt(mean(x^2) + eps) (one CTA).
__global__ void rms_scale_kernel(const float* __restrict__ x, int H, float eps,
                                 float* __restrict__ n) {
  __shared__ float red[32];
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) ss += x[i] * x[i];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
  const float r = 1.0f / sqrtf(tot / (float)H + eps);
  for (int i = threadIdx.x; i < H; i += blockDim.x) n[i] = x[i] * r;
}

// Weight multiply: n *= w (bf16).
__global__ void mul_kernel(float* __restrict__ n, const uint16_t* __restrict__ w, int H) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < H) n[i] *= __uint_as_float((uint32_t)w[i] << 16);
}

// y = W x, W bf16 row-major [N][K]; one warp per row, 16-byte loads.
__global__ void gemv_kernel(const uint16_t* __restrict__ W, int N, int K,
                            const float* __restrict__ x, float* __restrict__ y) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= N) return;
  const uint16_t* wr = W + (size_t)row * K;
  float acc = 0.f;
  for (int k = lane * 8; k < K; k += 256) {
    const uint4 w = *reinterpret_cast<const uint4*>(wr + k);
    acc = fmaf(bf16lo(w.x), x[k + 0], acc);
    acc = fmaf(bf16hi(w.x), x[k + 1], acc);
    acc = fmaf(bf16lo(w.y), x[k + 2], acc);
    acc = fmaf(bf16hi(w.y), x[k + 3], acc);
    acc = fmaf(bf16lo(w.z), x[k + 4], acc);
    acc = fmaf(bf16hi(w.z), x[k + 5], acc);
    acc = fmaf(bf16lo(w.w), x[k + 6], acc);
    acc = fmaf(bf16hi(w.w), x[k + 7], acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) y[row] = acc;
}

// RoPE on q (nq heads) and k (nkv heads) in place, rotate-half pairs.
__global__ void rope_kernel(float* __restrict__ q, float* __restrict__ k, int nq, int nkv, int hd,
                            const int* __restrict__ pos, const float2* __restrict__ tab,
                            int interleaved) {
  const int half = hd / 2;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int total = (nq + nkv) * half;
  if (idx >= total) return;
  const int head = idx / half, i = idx % half;
  float* v = head < nq ? q + (size_t)head * hd : k + (size_t)(head - nq) * hd;
  const float2 c = tab[(size_t)(*pos) * half + i];
  // pair i: dims (i, i + hd/2), or (2i, 2i + 1) when interleaved
  const int e = interleaved ? 2 * i : i, o = interleaved ? 2 * i + 1 : i + half;
  const float a = v[e], b = v[o];
  v[e] = a * c.x - b * c.y;
  v[o] = a * c.y + b * c.x;
}

// KV append: row pos of every KV head <- bf16(k), bf16(v).
__global__ void kv_append_kernel(const float* __restrict__ k, const float* __restrict__ v, int nkv,
                                 int hd, int max_ctx, const int* __restrict__ pos,
                                 uint16_t* __restrict__ kc, uint16_t* __restrict__ vc) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= nkv * hd) return;
  const int g = idx / hd, j = idx % hd;
  const size_t at = ((size_t)g * max_ctx + *pos) * hd + j;
  kc[at] = f32_to_bf16_bits(k[idx]);
  vc[at] = f32_to_bf16_bits(v[idx]);
}

// Attention of one query head (one CTA) over rows 0..pos of its KV head: each
// warp keeps a running max / sum / weighted V over its positions; warps merge.
template <int HD>
__global__ void attention_kernel(const float* __restrict__ q, const uint16_t* __restrict__ kc,
                                 const uint16_t* __restrict__ vc, int nq, int nkv, int max_ctx,
                                 const int* __restrict__ pos, float* __restrict__ o) {
  constexpr int DL = HD / 32;
  __shared__ float ws[8][HD + 2];
  const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = (int)((long)h * nkv / nq);
  const int n = *pos + 1;
  const float scale = rsqrtf((float)HD);
  float qr[DL], acc[DL];
  for (int j = 0; j < DL; ++j) {
    qr[j] = q[(size_t)h * HD + lane * DL + j] * scale;
    acc[j] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const uint16_t* K = kc + (size_t)g * max_ctx * HD;
  const uint16_t* V = vc + (size_t)g * max_ctx * HD;
  for (int t = warp; t < n; t += 8) {
    float d = 0.f;
    for (int j = 0; j < DL; ++j)
      d = fmaf(qr[j], __uint_as_float((uint32_t)K[(size_t)t * HD + lane * DL + j] << 16), d);
    d = warp_sum(d);
    const float mn = fmaxf(m, d);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - mn);
    const float p = expf(d - mn);
    l = l * alpha + p;
    for (int j = 0; j < DL; ++j)
      acc[j] = fmaf(p, __uint_as_float((uint32_t)V[(size_t)t * HD + lane * DL + j] << 16),
                    acc[j] * alpha);
    m = mn;
  }
  for (int j = 0; j < DL; ++j) ws[warp][lane * DL + j] = acc[j];
  if (lane == 0) {
    ws[warp][HD] = m;
    ws[warp][HD + 1] = l;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < HD; j += blockDim.x) {
    float M = -INFINITY;
    for (int w = 0; w < 8; ++w) M = fmaxf(M, ws[w][HD]);
    float A = 0.f, Ls = 0.f;
    for (int w = 0; w < 8; ++w) {
      const float e = (ws[w][HD] == -INFINITY) ? 0.f : expf(ws[w][HD] - M);
      A += ws[w][j] * e;
      Ls += ws[w][HD + 1] * e;
    }
    o[(size_t)h * HD + j] = A / Ls;
  }
}

// out = a + b (residual add); optional tap copy; optional position advance.
__global__ void add_kernel(const float* __restrict__ a, const float* __restrict__ b,
                           float* __restrict__ out, float* __restrict__ tap, int n,
                           int* pos_advance) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0 && pos_advance) atomicAdd(pos_advance, 1);
  if (i >= n) return;
  const float y = a[i] + b[i];
  out[i] = y;
  if (tap) tap[i] = y;
}

// a = silu(g) * u.
__global__ void swiglu_kernel(const float* __restrict__ g, const float* __restrict__ u,
                              float* __restrict__ a, int F) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < F) a[i] = g[i] / (1.0f + expf(-g[i])) * u[i];
}

// Per-32 absmax int8 quantisation (one warp per block): dx = amax / 127,
// q = round-half-even(z / dx) clamped to +-127, natural element order.
__global__ void quantize_kernel(const float* __restrict__ z, int K, int8_t* __restrict__ qx,
                                float* __restrict__ dx, int8_t* qtap, float* qstap) {
  const int blk = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (blk * 32 >= K) return;
  const float v = z[blk * 32 + lane];
  const float amax = warp_max(fabsf(v));
  const float d = __fdiv_rn(amax, 127.0f);
  int q = 0;
  if (d != 0.0f) {
    q = __float2int_rn(__fdiv_rn(v, d));
    q = q > 127 ? 127 : (q < -127 ? -127 : q);
  }
  qx[blk * 32 + lane] = (int8_t)q;
  if (lane == 0) dx[blk] = d;
  if (qtap) {
    qtap[blk * 32 + lane] = (int8_t)q;
    if (lane == 0) qstap[blk] = d;
  }
}

// y = W x for q4 weights in the ABI layout (nibbles [N][K/2], fp16 scales
// [N][K/32]) and int8 x with block scales: one warp per row, one lane per block.
__global__ void gemv_q4_kernel(const uint8_t* __restrict__ nib, const uint16_t* __restrict__ sc,
                               int N, int K, const int8_t* __restrict__ qx,
                               const float* __restrict__ dx, float* __restrict__ y) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= N) return;
  const int nb = K / 32;
  float acc = 0.f;
  for (int b = lane; b < nb; b += 32) {
    const uint4 w = *reinterpret_cast<const uint4*>(nib + (size_t)row * (K / 2) + b * 16);
    const uint4 xa = *reinterpret_cast<const uint4*>(qx + b * 32);
    const uint4 xb = *reinterpret_cast<const uint4*>(qx + b * 32 + 16);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    int dot = 0, xsum = 0;
    for (int i = 0; i < 4; ++i) {
      // weight word i holds elements 8i..8i+7: low nibbles the even ones
      const int even = (int)__byte_perm(xw[2 * i], xw[2 * i + 1], 0x6420);
      const int odd = (int)__byte_perm(xw[2 * i], xw[2 * i + 1], 0x7531);
      dot = __dp4a((int)(ww[i] & 0x0F0F0F0Fu), even, dot);
      dot = __dp4a((int)((ww[i] >> 4) & 0x0F0F0F0Fu), odd, dot);
      xsum = __dp4a(0x01010101, (int)xw[2 * i], xsum);
      xsum = __dp4a(0x01010101, (int)xw[2 * i + 1], xsum);
    }
    const float s = __half2float(__ushort_as_half(sc[(size_t)row * nb + b]));
    acc = fmaf(s * dx[b], (float)(dot - 8 * xsum), acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) y[row] = acc;
}

static inline int cdiv(int a, int b) { return (a + b - 1) / b; }

cudaError_t quantize(const float* z, int K, int8_t* qx, float* dx, int8_t* qtap, float* qstap,
                     cudaStream_t s) {
  quantize_kernel<<<cdiv(K / 32, 8), 256, 0, s>>>(z, K, qx, dx, qtap, qstap);
  return cudaGetLastError();
}
cudaError_t gemv_q4(const uint8_t* packed, const uint16_t* scales, int N, int K, const int8_t* qx,
                    const float* dx, float* y, cudaStream_t s) {
  gemv_q4_kernel<<<cdiv(N, 8), 256, 0, s>>>(packed, scales, N, K, qx, dx, y);
  return cudaGetLastError();
}

cudaError_t rms_scale(const float* x, int H, float eps, float* n, cudaStream_t s) {
  rms_scale_kernel<<<1, 1024, 0, s>>>(x, H, eps, n);
  return cudaGetLastError();
}
cudaError_t mul(float* n, const uint16_t* w, int H, cudaStream_t s) {
  mul_kernel<<<cdiv(H, 256), 256, 0, s>>>(n, w, H);
  return cudaGetLastError();
}
cudaError_t gemv(const uint16_t* W, int N, int K, const float* x, float* y, cudaStream_t s) {
  gemv_kernel<<<cdiv(N, 8), 256, 0, s>>>(W, N, K, x, y);
  return cudaGetLastError();
}
cudaError_t rope(float* q, float* k, int nq, int nkv, int hd, const int* pos, const float2* tab,
                 int interleaved,
                 cudaStream_t s) {
  rope_kernel<<<cdiv((nq + nkv) * hd / 2, 256), 256, 0, s>>>(q, k, nq, nkv, hd, pos, tab, interleaved);
  return cudaGetLastError();
}
cudaError_t kv_append(const float* k, const float* v, int nkv, int hd, int max_ctx, const int* pos,
                      uint16_t* kc, uint16_t* vc, cudaStream_t s) {
  kv_append_kernel<<<cdiv(nkv * hd, 256), 256, 0, s>>>(k, v, nkv, hd, max_ctx, pos, kc, vc);
  return cudaGetLastError();
}
cudaError_t attention(const float* q, const uint16_t* kc, const uint16_t* vc, int nq, int nkv,
                      int hd, int max_ctx, const int* pos, float* o, cudaStream_t s) {
  if (hd == 64)
    attention_kernel<64><<<nq, 256, 0, s>>>(q, kc, vc, nq, nkv, max_ctx, pos, o);
  else if (hd == 128)
    attention_kernel<128><<<nq, 256, 0, s>>>(q, kc, vc, nq, nkv, max_ctx, pos, o);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}
cudaError_t add(const float* a, const float* b, float* out, float* tap, int n, int* pos_advance,
                cudaStream_t s) {
  add_kernel<<<cdiv(n, 256), 256, 0, s>>>(a, b, out, tap, n, pos_advance);
  return cudaGetLastError();
}
cudaError_t swiglu(const float* g, const float* u, float* a, int F, cudaStream_t s) {
  swiglu_kernel<<<cdiv(F, 256), 256, 0, s>>>(g, u, a, F);
  return cudaGetLastError();
}

}  // namespace unf
}  // namespace tld
