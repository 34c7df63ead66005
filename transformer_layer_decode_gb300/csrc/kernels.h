// Parameter blocks and launchers of the decode kernels (host + device view).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace tld {

// Balanced contiguous split of `total` units over `parts`: part p owns
// [split_begin(p), split_begin(p+1)).
__host__ __device__ inline int64_t split_begin(int64_t total, int parts, int p) {
  return total * p / parts;
}
// The part owning unit u (inverse of split_begin).
// 32-bit forms, for total * parts < 2^31.
__host__ __device__ inline int split_begin32(int total, int parts, int p) { return total * p / parts; }
__host__ __device__ inline int split_owner32(int total, int parts, int u) {
  return ((u + 1) * parts - 1) / total;
}
__host__ __device__ inline int split_owner(int64_t total, int parts, int64_t u) {
  return (int)(((u + 1) * parts - 1) / total);
}

// ---- tiled weight layouts ---------------------------------------------------
// A [N][K] matrix is stored as row blocks of kTileR rows; each row block is a
// run of k-tiles (the last one narrower when K is not a multiple of the tile
// width), consecutive in memory in (row block, k-tile) order, so any range of
// tiles is one contiguous run of bytes: a CTA that owns a range of row blocks
// streams exactly one slab.
//   bf16: k-tiles of kTileK columns, row-major inside ([kTileR][kw] bf16).
//   q4:   k-tiles of kTileKQ4 columns (32 blocks of 32); inside, the packed
//         nibbles [kTileR][kw/2 bytes], then the fp16 scales [kw/32][kTileR].
constexpr int kTileR = 4;
constexpr int kTileK = 256;
constexpr int kTileKQ4 = 1024;
// Consumer warps of the GEMV kernels and of the fused phase kernels: one tile of
// each 16-tile stage per warp.  Sixteen keep enough warps in flight to hide the
// latency of the per-stage arithmetic (measured: 8 warps streamed the 7B-shape
// gate/up matrix at 5.4 TB/s, 16 at 5.9 TB/s, 4 at 4.3 TB/s).
#ifndef TLD_CONSUMER_WARPS
#define TLD_CONSUMER_WARPS 16
#endif
constexpr int kConsumerWarps = TLD_CONSUMER_WARPS;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // consumer warps + 1 producer warp
// Consumer warps of the standalone attention kernels, except the cluster
// kernels of GQA groups up to 2, which run 16 (larger groups need the register
// budget of 8 warps).
constexpr int kAttnWarps = 8;
// Shared memory budget per CTA.  Above half of the SM's 228 KB, so two CTAs of
// one kernel never share an SM; the next kernel (programmatic dependent launch)
// then takes each SM as soon as its current CTA leaves and starts streaming.
#ifndef TLD_SMEM_BUDGET_KB
#define TLD_SMEM_BUDGET_KB 220
#endif
constexpr int kSmemBudget = TLD_SMEM_BUDGET_KB * 1024;
constexpr int kAttnStageBytes = 32768;  // K chunk + V chunk, 16 KB each
// Online softmax: a head's reference max moves only when a score exceeds it by
// more than this (natural-log units: the weights stay below e^8 ~ 3e3).
constexpr float kAttnRescaleSlack = 8.f;
constexpr int kTimelineSlots = 8;       // u64 per launch of the timeline probe
// Most attention CTAs one KV head may be split over (bounds the merge).
constexpr int kMaxSplits = 32;
#ifndef TLD_COPIES_PER_STAGE
#define TLD_COPIES_PER_STAGE 4
#endif
#ifndef TLD_COPIES_PER_STAGE_Q4
#define TLD_COPIES_PER_STAGE_Q4 8
#endif
// bulk copies a GEMV stage is issued as (bf16, int4)
constexpr int kCopiesPerStage = TLD_COPIES_PER_STAGE;
constexpr int kCopiesPerStageQ4 = TLD_COPIES_PER_STAGE_Q4;
constexpr int kL2AheadBytes = 256 * 1024;  // L2 look-ahead per CTA and kernel
constexpr int kMaxCluster = 16;            // CTAs per KV head in the cluster attention
#ifndef TLD_STAGE_TILES
#define TLD_STAGE_TILES 16
#endif
constexpr int kStageTiles = TLD_STAGE_TILES;  // a GEMV stage: 16 tiles (32 KB bf16, 36 KB int4)
constexpr int kTilesPerWarp = kStageTiles / kConsumerWarps;
static_assert(kStageTiles % kConsumerWarps == 0, "every consumer warp takes whole tiles of a stage");
constexpr int kTileBytes = kTileR * kTileK * 2;                          // 2 KB
constexpr int kTileBytesQ4 = kTileR * (kTileKQ4 / 2 + kTileKQ4 / 16);    // 2304 B
constexpr int kStageBytes = kStageTiles * kTileBytes;                    // 32 KB
constexpr int kStageBytesQ4 = kStageTiles * kTileBytesQ4;                // 36 KB

// Byte geometry of one tiled matrix.
struct TileGeom {
  int K, tile_k, ktiles, kw_last;
  int64_t rb_bytes, tile_bytes;
  int stage_bytes;
  int copies;  // bulk copies a stage is issued as
};

__host__ __device__ inline TileGeom tile_geom(int K, bool q4) {
  TileGeom g;
  g.K = K;
  g.tile_k = q4 ? kTileKQ4 : kTileK;
  g.ktiles = (K + g.tile_k - 1) / g.tile_k;
  g.kw_last = K - g.tile_k * (g.ktiles - 1);
  g.rb_bytes = q4 ? (int64_t)kTileR * (K / 2 + K / 16) : (int64_t)kTileR * K * 2;
  g.tile_bytes = q4 ? kTileBytesQ4 : kTileBytes;
  g.stage_bytes = q4 ? kStageBytesQ4 : kStageBytes;
  g.copies = q4 ? kCopiesPerStageQ4 : kCopiesPerStage;
  return g;
}

__host__ __device__ inline int64_t tile_byte_offset(int64_t t, const TileGeom& g) {
  const int64_t rb = t / g.ktiles, kt = t - rb * g.ktiles;
  return rb * g.rb_bytes + kt * g.tile_bytes;
}

// bf16: element (row r, col k) inside the tiled layout (in elements).
__host__ __device__ inline int64_t tiled_elem_offset(int64_t r, int64_t k, int K) {
  const int ktiles = (K + kTileK - 1) / kTileK;
  const int64_t kt = k / kTileK;
  const int kw = (kt == ktiles - 1) ? K - kTileK * (ktiles - 1) : kTileK;
  return (r / kTileR) * (int64_t)kTileR * K + kt * (int64_t)kTileR * kTileK +
         (r % kTileR) * kw + (k - kt * kTileK);
}

// q4: byte of the packed pair (row r, columns 2c2 and 2c2+1).
__host__ __device__ inline int64_t q4_nibble_byte(int64_t r, int64_t c2, int K) {
  const TileGeom g = tile_geom(K, true);
  const int64_t kt = (2 * c2) / kTileKQ4;
  const int kw = (kt == g.ktiles - 1) ? g.kw_last : kTileKQ4;
  return (r / kTileR) * g.rb_bytes + kt * g.tile_bytes + (r % kTileR) * (kw / 2) +
         (c2 - kt * (kTileKQ4 / 2));
}

// q4: byte of the fp16 scale of (row r, block b).
__host__ __device__ inline int64_t q4_scale_byte(int64_t r, int64_t b, int K) {
  const TileGeom g = tile_geom(K, true);
  const int64_t kt = (32 * b) / kTileKQ4;
  const int kw = (kt == g.ktiles - 1) ? g.kw_last : kTileKQ4;
  return (r / kTileR) * g.rb_bytes + kt * g.tile_bytes + kTileR * (kw / 2) +
         ((b - kt * (kTileKQ4 / 32)) * kTileR + (r % kTileR)) * 2;
}

// ---- KV cache geometry ---------------------------------------------------------
// Contiguous: a layer's K (or V) cache is [nkv][max_ctx][hd].  Paged: it is a
// pool of pages [page][nkv][page_rows][hd] and a page table maps the chunk of
// positions [c * page_rows, (c + 1) * page_rows) to page pages[c] (the same
// table for every layer).  A page holds one attention chunk of one KV head, so
// an attention stage is one contiguous copy either way.
__host__ __device__ inline int64_t kv_row_offset(const int* pages, int page_rows, int nkv,
                                                 int max_ctx, int hd, int g, int t) {
  if (!pages) return ((int64_t)g * max_ctx + t) * hd;
  const int c = t / page_rows;
  return (((int64_t)pages[c] * nkv + g) * page_rows + (t - c * page_rows)) * hd;
}

// The next kernel's share of the bytes of one CTA index, fetched into L2 by
// that CTA's producer once its own stream is issued: HBM keeps streaming
// through the tail of a kernel (its last stages, epilogue, merge), when the
// next kernel's CTAs cannot start yet.  GEMV next: units are row blocks of
// unit_bytes at base.  Attention next: units are K/V chunks of the layer
// cache at kc / vc (kv != 0).
struct L2Ahead {
  const uint8_t* base;  // null: nothing to fetch
  const uint8_t* vbase;
  int64_t unit_bytes;
  int n_units, grid, cap;  // unit count, the next kernel's grid, bytes per CTA at most
  int kv, nkv, hd, max_ctx;
  const int* pos;
  int cluster;  // attention next: its cluster size (0: global-merge grid)
  const int* pages;  // paged KV cache: page table (null: contiguous)
};

// The int8 input of an int4 GEMV, quantized once by the kernel that produces
// the vector ("the norm writes the matmul's quantized input") instead of by
// every CTA of the GEMV.  Per 32-block: the codes in the dp4a arrangement, the
// block scale amax / 127 (for an RMSNorm input: of x * w, the GEMV applying
// the 1 / rms), the sum of the codes.  An RMSNorm input also gets one sum of
// squares per producing CTA, which the GEMV adds in CTA order.  A block cut
// between CTAs is quantized by the CTA that writes its last element (per-block
// count of elements written, taken modulo 32; the GEMV that reads the codes
// clears the counts for the next round).
struct QVec {
  uint8_t* codes;      // [K] (null: no published input / output)
  float* scale;        // [K / 32]
  int32_t* sum;        // [K / 32]
  float* part;         // [n_part] sums of squares, or null (not an RMSNorm input)
  unsigned* cnt;       // [K / 32] element counts, or null (blocks written whole)
  const uint16_t* w;   // producer side: bf16 RMSNorm weight multiplied in, or null
  int K, n_part;
};

enum Prologue : int { PRO_NORM = 0, PRO_PLAIN = 1 };
enum Epilogue : int { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LOGITS = 3 };

struct GemvParams {
  const uint8_t* w;  // tiled weights
  TileGeom geo;
  int n_rb, nstages, max_rb_local;
  // prologue
  const float* x;          // input vector [K]
  const uint16_t* norm_w;  // bf16 [K] (PRO_NORM)
  float eps;
  float* x_copy;           // if set, CTA 0 also copies x here
  int* err;
  // EPI_QKV: rows are q (pair-interleaved per head), k (same), v
  int nq, nkv, hd, max_ctx;
  int rope_inter;       // RoPE pairs (2i, 2i+1) (rows in ABI order) instead of (i, i+hd/2)
  const int* pos;       // device step position
  const float2* rope;   // [max_ctx][hd/2] (cos, sin)
  float* q_out;         // [nq*hd]
  uint16_t* kc;         // layer cache (kv_row_offset)
  uint16_t* vc;
  const int* pages;     // paged KV cache: page table (null: contiguous [nkv][max_ctx][hd])
  // EPI_RESID
  const float* resid;
  float* out;
  float* tap;
  int* pos_advance;     // if set, CTA 0 adds 1 here (end of a step)
  // EPI_SWIGLU: rows interleave gate and up
  float* a_out;
  uint64_t* tl;  // optional timeline probe (kTimelineSlots x u64)
  // q4 weights: the int8 input of this GEMV is also written here by CTA 0
  int8_t* qtap;    // [K] natural order, or null
  float* qstap;    // [K/32] block scales, or null
  int32_t* dots;   // [n_rb * kTileR][K/32] integer block dots (tiled row order), or null
  L2Ahead ahead;
  QVec qin;    // q4: the published int8 input (else this GEMV quantizes x itself)
  QVec qout;   // q4: publish the int8 quantization of this GEMV's output vector
};

struct AttnParams {
  const uint16_t* kc;  // layer cache (kv_row_offset)
  const uint16_t* vc;
  const int* pages;    // paged KV cache: page table (null: contiguous [nkv][max_ctx][hd])
  const float* q;      // [nq*hd] rotated
  float* o;            // [nq*hd]
  float* part;         // [grid][2][G][hd+4]: (acc, m, l) of split heads
  int* counters;       // [nkv] arrivals per split head, zero between launches
  const int* pos;
  int* err;
  int nkv, max_ctx, nstages;
  float scale;
  uint64_t* tl;  // optional timeline probe (kTimelineSlots x u64)
  L2Ahead ahead;
  int cluster;   // > 0: grid = nkv clusters of this many CTAs, merged in shared memory
  QVec qout;     // q4 layer: publish the int8 quantization of o (blocks written whole)
};

// ---- two-phase kernels of the three-kernel layer ------------------------------
// One launch runs two phases separated by a grid barrier; the producer streams
// the second phase's bytes right after the first's, so HBM keeps streaming
// while the consumers finish the first phase and wait at the barrier.  Every
// CTA is resident (one CTA per SM, grid = SM count).  Barrier counters: two per
// launch site, alternating by the parity of the step position (the other one
// is cleared for the next step).
struct AttnOprojParams {  // attention (flat grid, global merge), then o-proj + residual
  AttnParams attn;
  GemvParams o;
  int* bar;               // [2] barrier counters of this launch site
  int att_grid;           // CTAs taking part in the attention phase (<= grid)
  int nstages, slot_bytes;
  uint64_t* tl2;          // timeline row of the o-proj phase or null
};

struct FfnParams {  // norm + gate/up + SwiGLU, then down + residual
  GemvParams gu, down;
  int* bar;
  int nstages, slot_bytes;
  uint64_t* tl2;          // timeline row of the down phase or null
};

// Attention with the o-projection split by KV-head group, in one cluster
// launch: cluster g (C CTAs) attends for the query heads of KV head g, merges
// them in distributed shared memory, and every CTA of the cluster receives the
// group's whole output o_g (G * hd values).  CTA rank r then multiplies o_g by
// rows [rb0, rb1) of Wo_g = Wo[:, g*G*hd : (g+1)*G*hd] (the columns of the
// group, stored per group in the tiled layout of K = G*hd), streamed right
// behind its K/V chunks, into part[g][rows].  The CTA of rank r that finishes
// last among the nkv clusters adds the nkv partial vectors of its rows in
// group order to the residual: out = resid + sum_g Wo_g o_g.
struct AttnHeadProjParams {
  AttnParams attn;        // cluster attention (attn.cluster = C CTAs per KV head)
  const uint8_t* wo;      // group g's tiled Wo_g at wo + g * group_bytes
  int64_t group_bytes;
  TileGeom geo;           // of K = G * hd
  int n_rb;               // hidden / 4 row blocks per group
  const float* resid;     // [hidden]
  float* out;             // [hidden]
  float* tap;             // optional copy of out
  float* part;            // [nkv][hidden] per-group partial projections
  int* cnt;               // [C] arrivals per row range (zero between launches)
  int nstages, slot_bytes;
  uint64_t* tl2;          // timeline row of the projection phase or null
  L2Ahead ahead;          // the next kernel's bytes
  int8_t* qtap;           // q4: the int8 o (natural order) and its block scales, or null
  float* qstap;
  int32_t* dots;          // q4: [hidden][G*hd*nkv/32] integer block dots, or null
};
size_t attn_headproj_smem_bytes(int hd, int G, bool q4, int nstages, int quads, int nkv);
const void* attn_headproj_kernel_ptr(int hd, int G, bool q4);
cudaError_t launch_attn_headproj(int hd, int G, bool q4, const AttnHeadProjParams& p, int grid,
                                 size_t smem, cudaStream_t s, bool pdl);
cudaError_t launch_repack_groups(const void* src, bool q4_scales, bool q4, int rows, int K, int Kg,
                                 uint8_t* dst, int64_t group_bytes, cudaStream_t s);

// The LM head after the stack: final RMSNorm x weight + vocabulary GEMV
// (PRO_NORM, EPI_LOGITS: rows to g.out) and the greedy token.
struct LmHeadParams {
  GemvParams g;
  unsigned long long* key;  // [2]: best key of the running launch, CTA ticket (both zero between launches)
  int* token_out;           // device int32: the chosen row
};
cudaError_t launch_lm_head(const LmHeadParams& p, int grid, size_t smem, cudaStream_t s, bool pdl);
const void* lm_head_kernel_ptr();

size_t attn_oproj_smem_bytes(int hd, int G, int K_o, int max_rb_o, bool q4, int nstages,
                             int slot_bytes);
size_t ffn_smem_bytes(int K_gu, int max_rb_gu, int K_down, int max_rb_down, bool q4, int nstages,
                      int slot_bytes);
const void* attn_oproj_kernel_ptr(int hd, int G, bool q4);
const void* ffn_kernel_ptr(bool q4);
cudaError_t launch_attn_oproj(int hd, int G, bool q4, const AttnOprojParams& p, int grid,
                              size_t smem, cudaStream_t s, bool pdl);
cudaError_t launch_ffn(bool q4, const FfnParams& p, int grid, size_t smem, cudaStream_t s,
                       bool pdl);

// ---- the persistent per-token kernel ---------------------------------------
struct PLayer {  // per-layer pointers
  const uint8_t* wqkv;
  const uint8_t* wo;
  const uint8_t* wgu;
  const uint8_t* wd;
  const uint16_t* attn_norm;
  const uint16_t* ffn_norm;
  uint16_t* kc;
  uint16_t* vc;
};

struct TokenParams {
  const PLayer* layers;  // device [n_layers]
  int n_layers, hidden;
  // parameter templates of the phases (shapes, geometry, workspace pointers);
  // the per-layer and per-step pointers are filled in by the kernel
  GemvParams qkv, o, gu, down;
  AttnParams attn;
  int att_grid;          // CTAs taking part in the attention phase
  const float* emb;      // step input
  float* out;            // step output
  float* X;              // residual stream between layers
  float* tap;            // per-layer outputs [n_layers][hidden] or null
  int* pos;              // device step position (read at start, +1 at the end)
  int* bar;              // two grid-barrier counters, alternating by position parity
  int* err;
  int nstages, slot_bytes;
  int8_t* qtap;          // int8 GEMV-input taps [n_layers][4][km] or null
  float* qstap;
  int km;
  int32_t* dots;         // block-dot tap of one GEMV or null
  int dot_layer, dot_kernel;
  uint64_t* tl;          // timeline probe [5 * n_layers][kTimelineSlots] or null
};

size_t persistent_work_bytes(const TokenParams& P, int hd, int G, bool q4);
const void* persistent_kernel_ptr(int hd, int G, bool q4);
// Cooperative launch (all CTAs resident) of the persistent kernel.
cudaError_t launch_persistent(int hd, int G, bool q4, const TokenParams& P, int grid, size_t smem,
                              cudaStream_t s);

// Shared memory the fused kernels need.
size_t gemv_smem_bytes(int K, bool q4, int nstages, int max_rb_local);
size_t attn_smem_bytes(int hd, int G, int nstages, bool cluster = false);
int attn_consumer_warps(int hd, int G, bool cluster);

// Launch with programmatic stream serialization (the kernel may start while
// the previous one on the stream finishes; it waits before reading its inputs).
cudaError_t launch_gemv(int pro, int epi, bool q4, const GemvParams& p, int grid, size_t smem,
                        cudaStream_t s, bool pdl);
// p.cluster > 0: a cluster launch, grid = nkv * p.cluster.
cudaError_t launch_attn(int hd, int G, const AttnParams& p, int grid, size_t smem,
                        cudaStream_t s, bool pdl);
const void* attn_kernel_ptr(int hd, int G, bool cluster);
const void* gemv_kernel_ptr(int pro, int epi, bool q4);
cudaError_t set_smem_limits();
// Error flag of dec_attention_noalloc on the current device (see dec_sync_status).
int noalloc_sync_status(cudaStream_t stream, int* flag_out);

// Load-time repack of a row-major [rows][K] bf16 block into the tiled layout
// of a matrix with K columns, source row s going to tiled row map(s):
//   map = dst_row0 + s                                  (kind 0, plain; also
//                                                        q/k rows whose RoPE
//                                                        pairs are (2i, 2i+1))
//   q/k heads: dst_row0 + rope pair interleave          (kind 1: pairs (i, i+hd/2)
//                                                        made adjacent)
//   gate/up:   dst_row0 + 2*s (+1 for up via dst_row0)  (kind 2)
cudaError_t launch_repack_bf16(const uint16_t* src, int rows, int K, uint8_t* dst_tiled,
                               int dst_row0, int kind, int hd, cudaStream_t s);
// The same row maps for q4 weights: packed nibbles [rows][K/2] and fp16 scales
// [rows][K/32] into the q4 tiled layout.
cudaError_t launch_repack_q4(const uint8_t* nibbles, const uint16_t* scales, int rows, int K,
                             uint8_t* dst_tiled, int dst_row0, int kind, int hd, cudaStream_t s);

// ---- the unfused plan: one kernel per op -------------------------------------
namespace unf {
cudaError_t rms_scale(const float* x, int H, float eps, float* n, cudaStream_t s);
cudaError_t mul(float* n, const uint16_t* w, int H, cudaStream_t s);
cudaError_t gemv(const uint16_t* W, int N, int K, const float* x, float* y, cudaStream_t s);
cudaError_t rope(float* q, float* k, int nq, int nkv, int hd, const int* pos, const float2* tab,
                 int interleaved, cudaStream_t s);
cudaError_t kv_append(const float* k, const float* v, int nkv, int hd, int max_ctx, const int* pos,
                      uint16_t* kc, uint16_t* vc, cudaStream_t s);
cudaError_t attention(const float* q, const uint16_t* kc, const uint16_t* vc, int nq, int nkv,
                      int hd, int max_ctx, const int* pos, float* o, cudaStream_t s);
cudaError_t add(const float* a, const float* b, float* out, float* tap, int n, int* pos_advance,
                cudaStream_t s);
cudaError_t swiglu(const float* g, const float* u, float* a, int F, cudaStream_t s);
// q4 path: per-32 absmax int8 quantization of z; GEMV on ABI-layout q4 weights.
cudaError_t quantize(const float* z, int K, int8_t* qx, float* dx, int8_t* qtap, float* qstap,
                     cudaStream_t s);
cudaError_t gemv_q4(const uint8_t* packed, const uint16_t* scales, int N, int K, const int8_t* qx,
                    const float* dx, float* y, cudaStream_t s);
}  // namespace unf

}  // namespace tld
