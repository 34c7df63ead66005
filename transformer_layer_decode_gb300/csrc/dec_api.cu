// C ABI of the decode library: validation, device memory, the per-layer launch
// plan (fused or unfused), and the whole-token CUDA graph whose only
// per-step change is the step position held in device memory ("Vulkan Command
// Buffer Reuse vs CUDA Graphs: RDNA4 Decode Overhead", section "Why NVIDIA got
// a free 14 percent": capture once, patch the few per-token parameters).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/dec.h"
#include "common.cuh"
#include "kernels.h"

using namespace tld;

namespace {

constexpr int kNumMats = 7;  // q k v o gate up down

struct Tiled {  // one fused-plan matrix in the tiled layout
  uint8_t* w = nullptr;
  TileGeom geo{};
  int N = 0, K = 0, n_rb = 0, nstages = 0, max_rb_local = 0;
  size_t bytes = 0, smem = 0;
};

struct LayerDev {
  uint16_t* attn_norm = nullptr;
  uint16_t* ffn_norm = nullptr;
  Tiled qkv, o, gu, down;                       // fused plan
  uint16_t* mats[kNumMats] = {};                // unfused plan: row-major bf16
  uint8_t* q4n[kNumMats] = {};                  // unfused plan: q4 nibbles [N][K/2]
  uint16_t* q4s[kNumMats] = {};                 // unfused plan: q4 scales [N][K/32]
  uint16_t* kc = nullptr;
  uint16_t* vc = nullptr;
  uint32_t loaded = 0;                          // bit per tensor id
  int kv_len = 0;
};

thread_local std::string g_create_error;

}  // namespace

struct dec_handle {
  dec_model_desc d{};
  int n_sm = 0, G = 0;
  bool fused = true, graph = true, pdl = true, persistent = false, l2_ahead = true;
  bool cluster_attn = true;
  bool three = false;  // fused plan: three kernels per layer (else five)
  bool four = false;   // fused plan: QKV, attention, o-proj, gate/up + down
  bool rope_inter = false;  // RoPE pairs (2i, 2i+1)
  // paged KV cache: pages of page_rows positions of one KV head; the page table
  // (host copy and device copy) maps position chunk c to page pages[c]
  bool paged = false;
  int page_rows = 0, n_pages = 0;
  std::vector<int> h_pages;
  int* d_pages = nullptr;
  // three-kernel plan: barrier counters [n_layers][2 launch sites][2 parities],
  // and the ring / shared memory of the two-phase kernels
  int* d_fbar = nullptr;
  int ao_nstages = 0, ao_slot = 0, ffn_nstages = 0, ffn_slot = 0;
  size_t ao_smem = 0, ffn_smem = 0;
  std::vector<LayerDev> layers;
  std::vector<void*> allocs;
  // DEC_DEBUG_GUARDS: every allocation sits between guard bands of a known
  // byte pattern, checked by dec_check_guards
  bool guards = false;
  struct Guard {
    uint8_t* user;  // start of the caller-visible bytes
    size_t bytes;
  };
  std::vector<Guard> guard_list;
  // activations / workspace
  float *X = nullptr, *h1 = nullptr, *q = nullptr, *o = nullptr, *a = nullptr;
  float *n1 = nullptr, *k = nullptr, *v = nullptr, *g = nullptr, *u = nullptr, *y = nullptr;
  int8_t* qbuf = nullptr;  // unfused q4: int8 GEMV input
  float* dbuf = nullptr;   // and its block scales
  // persistent plan
  PLayer* d_players = nullptr;
  int* d_bar = nullptr;
  int p_nstages = 0, p_slot = 0;
  size_t p_smem = 0;
  // int4 weights, five- and four-kernel plans: each GEMV's int8 input is
  // published once by the kernel that produces the vector (QVec): the inputs
  // of the QKV (n1), o-proj (o), gate/up (n2) and down (a) projections
  bool qpub = false;
  // attention + o-projection by KV-head group in one cluster launch
  // (DEC_FUSE_ATTN_OPROJ): Wo stored per group, the groups' partial vectors,
  // arrival counters per row range
  bool headproj = false;
  TileGeom hp_geo{};
  int64_t hp_group_bytes = 0;
  int hp_nstages = 0;
  size_t hp_smem = 0;
  float* hp_part = nullptr;
  int* hp_cnt = nullptr;
  enum { QS_N1 = 0, QS_O = 1, QS_N2 = 2, QS_A = 3 };
  QVec qs[4] = {};
  float* apart = nullptr;  // attention partial records
  int* acount = nullptr;   // attention arrivals per split head
  int att_grid = 0;
  int att_cluster = 0;  // fused plan: CTAs per KV head (cluster merge); 0 = global merge
  int* d_pos = nullptr;
  int* d_err = nullptr;
  float2* rope = nullptr;
  uint16_t* staging = nullptr;
  size_t staging_bytes = 0;
  size_t attn_smem = 0;
  int attn_nstages = 0;
  int kv_len = 0;
  int64_t weight_bytes = 0, kv_bytes = 0, ws_bytes = 0;
  // taps
  uint64_t* timeline = nullptr;
  int32_t* dot_tap = nullptr;
  int dot_layer = -1, dot_kernel = -1;
  float* tap = nullptr;
  int8_t* qtap = nullptr;
  float* qstap = nullptr;
  // LM head after the stack (optional)
  Tiled lm;
  uint16_t* lm_norm = nullptr;
  float* logits = nullptr;             // [vocab], when the caller gives no tap
  unsigned long long* lm_key = nullptr;  // [2]: running best key, CTA ticket
  int vocab = 0;
  bool lm_loaded = false;
  int32_t* token_out = nullptr;
  float* logits_tap = nullptr;
  cudaGraphNode_t lm_node = nullptr;
  // graph
  cudaStream_t cap_stream = nullptr;
  cudaGraph_t graph_g = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t first_node = nullptr, last_node = nullptr;
  const float* cap_emb = nullptr;
  float* cap_out = nullptr;
  std::string err;
};

namespace {

int fail(dec_handle* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->err = buf;
  else g_create_error = buf;
  return code;
}

int cuda_fail(dec_handle* h, cudaError_t e, const char* what) {
  return fail(h, DEC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define TLD_CUDA(h, call)                                    \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return cuda_fail((h), e_, #call); \
  } while (0)

constexpr size_t kGuardBytes = 256;      // guard band on each side (keeps 256-byte alignment)
constexpr uint8_t kGuardPattern = 0xA5;

template <class T>
int dev_alloc(dec_handle* h, T** p, size_t bytes, int64_t* account) {
  void* v = nullptr;
  const size_t user = bytes < 16 ? 16 : bytes;
  const size_t total = h->guards ? user + 2 * kGuardBytes + 255 : user;
  cudaError_t e = cudaMalloc(&v, total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(h, DEC_ERR_OOM, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
  }
  h->allocs.push_back(v);
  if (account) *account += (int64_t)bytes;
  if (h->guards) {
    // [guard | user bytes | pattern up to the next 256 and a guard]; the user
    // bytes start poisoned (0xFF: NaN as fp32 and as bf16) so that a read of
    // a byte nothing wrote shows up in the results
    uint8_t* base = static_cast<uint8_t*>(v);
    e = cudaMemset(base, kGuardPattern, total);
    if (e == cudaSuccess) e = cudaMemset(base + kGuardBytes, 0xFF, user);
    if (e != cudaSuccess) return cuda_fail(h, e, "guard bands");
    h->guard_list.push_back({base + kGuardBytes, user});
    *p = reinterpret_cast<T*>(base + kGuardBytes);
    return DEC_OK;
  }
  *p = static_cast<T*>(v);
  return DEC_OK;
}

// Plans one tiled matrix: each CTA owns whole row blocks; the ring gets as
// many stages as the shared-memory budget leaves.
void plan_tiled(Tiled& t, int N, int K, int n_sm, bool q4) {
  t.N = N;
  t.K = K;
  t.geo = tile_geom(K, q4);
  t.n_rb = N / kTileR;
  t.bytes = (size_t)t.n_rb * t.geo.rb_bytes;
  t.max_rb_local = (t.n_rb + n_sm - 1) / n_sm;
  const size_t fixed = gemv_smem_bytes(K, q4, 0, t.max_rb_local);
  int ns = (int)(((size_t)kSmemBudget > fixed ? kSmemBudget - fixed : 0) / t.geo.stage_bytes);
  if (ns < 2) ns = 2;
  if (ns > 8) ns = 8;
  t.nstages = ns;
  t.smem = gemv_smem_bytes(K, q4, ns, t.max_rb_local);
}

int max_k(const dec_model_desc& d) {
  int m = d.hidden;
  if (d.ffn > m) m = d.ffn;
  if (d.n_q_heads * d.head_dim > m) m = d.n_q_heads * d.head_dim;
  return m;
}

void mat_shape(const dec_model_desc& d, int tensor, int* N, int* K) {
  const int H = d.hidden, hd = d.head_dim, F = d.ffn;
  switch (tensor) {
    case DEC_T_WQ: *N = d.n_q_heads * hd; *K = H; break;
    case DEC_T_WK: *N = d.n_kv_heads * hd; *K = H; break;
    case DEC_T_WV: *N = d.n_kv_heads * hd; *K = H; break;
    case DEC_T_WO: *N = H; *K = d.n_q_heads * hd; break;
    case DEC_T_WGATE: *N = F; *K = H; break;
    case DEC_T_WUP: *N = F; *K = H; break;
    case DEC_T_WDOWN: *N = H; *K = F; break;
    default: *N = *K = 0;
  }
}

uint32_t required_mask(const dec_model_desc& d) {
  uint32_t m = (1u << DEC_T_ATTN_NORM) | (1u << DEC_T_FFN_NORM);
  for (int t = DEC_T_WQ; t <= DEC_T_WDOWN; ++t) {
    if (t == DEC_T_FFN_NORM) continue;
    m |= 1u << t;
    if (d.weight_fmt == DEC_W_Q4B32) m |= 1u << (t + DEC_T_SCALES);
  }
  return m;
}

// Index 0..6 of a matrix tensor id (q k v o gate up down).
int mat_index(int tensor) { return tensor <= DEC_T_WO ? tensor - DEC_T_WQ : tensor - DEC_T_WQ - 1; }

void drop_graph(dec_handle* h) {
  if (h->exec) cudaGraphExecDestroy(h->exec);
  if (h->graph_g) cudaGraphDestroy(h->graph_g);
  h->exec = nullptr;
  h->graph_g = nullptr;
  h->first_node = h->last_node = h->lm_node = nullptr;
}

// Calls fn(element offset, rows, src row offset) for every run of rows
// [t0, t1) of every KV head that is contiguous in the cache layout (one run a
// head when contiguous, one a page when paged); the source row offset counts
// rows of a [nkv][t1 - t0][hd] array.
template <class Fn>
int for_kv_runs(const dec_handle* h, int t0, int t1, Fn&& fn) {
  const dec_model_desc& d = h->d;
  const int* pages = h->paged ? h->h_pages.data() : nullptr;
  for (int g = 0; g < d.n_kv_heads; ++g)
    for (int t = t0; t < t1;) {
      const int end = h->paged ? std::min(t1, (t / h->page_rows + 1) * h->page_rows) : t1;
      const int64_t off = kv_row_offset(pages, h->page_rows, d.n_kv_heads, d.max_ctx, d.head_dim, g, t);
      const int rc = fn(off, end - t, (int64_t)g * (t1 - t0) + (t - t0));
      if (rc) return rc;
      t = end;
    }
  return DEC_OK;
}

// ---- the fused plan ------------------------------------------------------------

// Launches per layer of a fused (non-persistent) plan.
int kernels_per_layer(const dec_handle* h) {
  if (h->three) return 3;
  return 5 - (h->four ? 1 : 0) - (h->headproj ? 1 : 0);
}

GemvParams gemv_base(const dec_handle* h, const Tiled& t) {
  GemvParams p{};
  p.w = t.w;
  p.geo = t.geo;
  p.n_rb = t.n_rb;
  p.nstages = t.nstages;
  p.max_rb_local = t.max_rb_local;
  p.eps = h->d.rms_eps;
  p.err = h->d_err;
  p.nq = h->d.n_q_heads;
  p.nkv = h->d.n_kv_heads;
  p.hd = h->d.head_dim;
  p.max_ctx = h->d.max_ctx;
  p.pos = h->d_pos;
  p.rope = h->rope;
  p.rope_inter = h->rope_inter ? 1 : 0;
  p.pages = h->paged ? h->d_pages : nullptr;
  return p;
}

GemvParams k1_params(const dec_handle* h, int l, const float* x_in, bool first) {
  const LayerDev& L = h->layers[l];
  GemvParams p = gemv_base(h, L.qkv);
  p.x = x_in;
  p.norm_w = L.attn_norm;
  p.x_copy = first ? h->X : nullptr;
  p.q_out = h->q;
  p.kc = L.kc;
  p.vc = L.vc;
  return p;
}

AttnParams k2_params(const dec_handle* h, int l) {
  const LayerDev& L = h->layers[l];
  AttnParams p{};
  p.kc = L.kc;
  p.vc = L.vc;
  p.pages = h->paged ? h->d_pages : nullptr;
  p.q = h->q;
  p.o = h->o;
  p.part = h->apart;
  p.counters = h->acount;
  p.pos = h->d_pos;
  p.err = h->d_err;
  p.nkv = h->d.n_kv_heads;
  p.max_ctx = h->d.max_ctx;
  p.nstages = h->attn_nstages;
  p.scale = (float)(1.0 / std::sqrt((double)h->d.head_dim));
  return p;
}

// The fused plan's attention grid: nkv clusters, or the global-merge grid.
int fused_att_grid(const dec_handle* h) {
  return h->att_cluster > 0 ? h->d.n_kv_heads * h->att_cluster : h->att_grid;
}

GemvParams k3_params(const dec_handle* h, int l) {
  GemvParams p = gemv_base(h, h->layers[l].o);
  p.x = h->o;
  p.resid = h->X;
  p.out = h->h1;
  return p;
}

GemvParams k4_params(const dec_handle* h, int l) {
  const LayerDev& L = h->layers[l];
  GemvParams p = gemv_base(h, L.gu);
  p.x = h->h1;
  p.norm_w = L.ffn_norm;
  p.a_out = h->a;
  return p;
}

GemvParams k5_params(const dec_handle* h, int l, float* out, bool last_of_step) {
  GemvParams p = gemv_base(h, h->layers[l].down);
  p.x = h->a;
  p.resid = h->h1;
  p.out = out;
  p.tap = h->tap ? h->tap + (size_t)l * h->d.hidden : nullptr;
  p.pos_advance = last_of_step ? h->d_pos : nullptr;
  return p;
}

cudaGraphNode_t last_captured_node(cudaStream_t s) {
  cudaStreamCaptureStatus st;
  const cudaGraphNode_t* deps = nullptr;
  size_t n = 0;
  if (cudaStreamGetCaptureInfo(s, &st, nullptr, nullptr, &deps, nullptr, &n) != cudaSuccess ||
      st != cudaStreamCaptureStatusActive || n == 0)
    return nullptr;
  return deps[n - 1];
}

// What kernel `kernel` of layer l prefetches into L2 for the kernel after it.
L2Ahead l2_ahead_of(const dec_handle* h, int kernel, int l) {
  L2Ahead a{};
  if (!h->l2_ahead) return a;
  const LayerDev& L = h->layers[l];
  auto rows = [&](const Tiled& t) {
    a.base = t.w;
    a.unit_bytes = t.geo.rb_bytes;
    a.n_units = t.n_rb;
    a.grid = h->n_sm;
    a.cap = kL2AheadBytes;
  };
  switch (kernel) {
    case 0:  // attention reads this layer's K/V
      a.kv = 1;
      a.base = reinterpret_cast<const uint8_t*>(L.kc);
      a.vbase = reinterpret_cast<const uint8_t*>(L.vc);
      a.nkv = h->d.n_kv_heads;
      a.hd = h->d.head_dim;
      a.max_ctx = h->d.max_ctx;
      a.pos = h->d_pos;
      a.grid = fused_att_grid(h);
      a.cluster = h->att_cluster;
      a.pages = h->paged ? h->d_pages : nullptr;
      a.cap = kL2AheadBytes;
      break;
    case 1: rows(L.o); break;
    case 2: rows(L.gu); break;
    case 3: rows(L.down); break;
    default: rows(h->layers[(l + 1) % h->d.n_layers].qkv); break;  // the next layer (or token)
  }
  return a;
}

// Parameters of fused GEMV kernel `kernel` (0: QKV, 2: o-proj, 3: gate/up,
// 4: down) of layer l.  in_step: part of a dec_step (first / last layer I/O,
// taps, timeline); otherwise a standalone launch on the workspaces.  The graph
// capture and the later pointer patching both build their nodes from here.
GemvParams fused_gemv_params(const dec_handle* h, int kernel, int l, const float* emb, float* out,
                             bool in_step) {
  const bool first = in_step && l == 0;
  const bool last = l == h->d.n_layers - 1;
  GemvParams p{};
  int slot = 0;
  switch (kernel) {
    case 0: p = k1_params(h, l, first ? emb : h->X, first); slot = 0; break;
    case 2: p = k3_params(h, l); slot = 1; break;
    case 3: p = k4_params(h, l); slot = 2; break;
    default: p = k5_params(h, l, (in_step && last) ? out : h->X, in_step && last); slot = 3; break;
  }
  p.tl = (in_step && h->timeline) ? h->timeline + kTimelineSlots * (size_t)(l * 5 + kernel) : nullptr;
  p.ahead = l2_ahead_of(h, kernel, l);
  if (in_step && h->qtap) {  // int8 input taps: q, o, gate and down projections of layer l
    const int km = max_k(h->d);
    p.qtap = h->qtap + ((size_t)l * 4 + slot) * km;
    p.qstap = h->qstap + ((size_t)l * 4 + slot) * (km / 32);
  }
  if (in_step && h->dot_tap && h->dot_layer == l && h->dot_kernel == kernel) p.dots = h->dot_tap;
  if (h->qpub) {  // published int8 inputs (the first layer's QKV quantizes its input itself)
    const QVec* q = h->qs;
    switch (kernel) {
      case 0:
        if (l > 0) p.qin = q[dec_handle::QS_N1];
        break;
      case 2:
        p.qin = q[dec_handle::QS_O];
        p.qout = q[dec_handle::QS_N2];
        p.qout.w = h->layers[l].ffn_norm;
        break;
      case 3:
        p.qin = q[dec_handle::QS_N2];
        p.qout = q[dec_handle::QS_A];
        break;
      default:
        p.qin = q[dec_handle::QS_A];
        if (!last) {
          p.qout = q[dec_handle::QS_N1];
          p.qout.w = h->layers[l + 1].attn_norm;
        }
        break;
    }
  }
  return p;
}

AttnHeadProjParams hp_params(const dec_handle* h, int l, bool in_step) {
  const LayerDev& L = h->layers[l];
  AttnHeadProjParams p{};
  p.attn = k2_params(h, l);
  p.attn.tl = (in_step && h->timeline) ? h->timeline + kTimelineSlots * (size_t)(l * 5 + 1) : nullptr;
  p.attn.cluster = h->att_cluster;
  p.wo = L.o.w;
  p.group_bytes = h->hp_group_bytes;
  p.geo = h->hp_geo;
  p.n_rb = h->d.hidden / kTileR;
  p.resid = h->X;
  p.out = h->h1;
  p.part = h->hp_part;
  p.cnt = h->hp_cnt;
  p.nstages = h->hp_nstages;
  p.slot_bytes = kAttnStageBytes;
  p.tl2 = (in_step && h->timeline) ? h->timeline + kTimelineSlots * (size_t)(l * 5 + 2) : nullptr;
  p.ahead = l2_ahead_of(h, 2, l);  // the gate/up weights
  if (in_step && h->qtap) {  // the o-projection's int8 input (slot 1 of the layer's taps)
    const int km = max_k(h->d);
    p.qtap = h->qtap + ((size_t)l * 4 + 1) * km;
    p.qstap = h->qstap + ((size_t)l * 4 + 1) * (km / 32);
  }
  if (in_step && h->dot_tap && h->dot_layer == l && h->dot_kernel == 2) p.dots = h->dot_tap;
  return p;
}

AttnOprojParams ao_params(const dec_handle* h, int l, const float* emb, float* out, bool in_step) {
  AttnOprojParams p{};
  p.attn = k2_params(h, l);
  p.attn.tl = (in_step && h->timeline) ? h->timeline + kTimelineSlots * (size_t)(l * 5 + 1) : nullptr;
  p.o = fused_gemv_params(h, 2, l, emb, out, in_step);
  p.tl2 = p.o.tl;
  p.bar = h->d_fbar + (size_t)l * 4;
  p.att_grid = h->att_grid;
  p.nstages = h->ao_nstages;
  p.slot_bytes = h->ao_slot;
  return p;
}

FfnParams ffn_params(const dec_handle* h, int l, const float* emb, float* out, bool in_step) {
  FfnParams p{};
  p.gu = fused_gemv_params(h, 3, l, emb, out, in_step);
  p.down = fused_gemv_params(h, 4, l, emb, out, in_step);
  p.tl2 = p.down.tl;
  p.bar = h->d_fbar + (size_t)l * 4 + 2;
  p.nstages = h->ffn_nstages;
  p.slot_bytes = h->ffn_slot;
  return p;
}

int enqueue_fused_kernel(dec_handle* h, int kernel, int l, const float* emb, float* out,
                         bool in_step, cudaStream_t s) {
  const int nb = h->n_sm;
  const LayerDev& L = h->layers[l];
  const bool q4 = h->d.weight_fmt == DEC_W_Q4B32;
  cudaError_t e = cudaSuccess;
  if (h->headproj) {
    // QKV; attention + o-projection; then gate/up and down, or the two-phase FFN
    if (kernel == 1) {
      e = launch_attn_headproj(h->d.head_dim, h->G, q4, hp_params(h, l, in_step), fused_att_grid(h),
                               h->hp_smem, s, h->pdl);
      if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
      return DEC_OK;
    }
    if (kernel >= kernels_per_layer(h)) return fail(h, DEC_ERR_ARG, "kernel id %d out of range", kernel);
    if (kernel >= 2) kernel = h->four ? 3 : kernel + 1;  // the five-kernel plan's ids
  }
  if (h->four && kernel == 3) {
    e = launch_ffn(q4, ffn_params(h, l, emb, out, in_step), nb, h->ffn_smem, s, h->pdl);
    if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
    return DEC_OK;
  }
  if (h->four && kernel > 3) return fail(h, DEC_ERR_ARG, "kernel id %d out of range", kernel);
  if (h->three) {
    switch (kernel) {
      case 0:
        e = launch_gemv(PRO_NORM, EPI_QKV, q4, fused_gemv_params(h, 0, l, emb, out, in_step), nb,
                        L.qkv.smem, s, h->pdl);
        break;
      case 1:
        e = launch_attn_oproj(h->d.head_dim, h->G, q4, ao_params(h, l, emb, out, in_step), nb,
                              h->ao_smem, s, h->pdl);
        break;
      case 2:
        e = launch_ffn(q4, ffn_params(h, l, emb, out, in_step), nb, h->ffn_smem, s, h->pdl);
        break;
      default:
        return fail(h, DEC_ERR_ARG, "kernel id %d out of range", kernel);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
    return DEC_OK;
  }
  switch (kernel) {
    case 0:
      e = launch_gemv(PRO_NORM, EPI_QKV, q4, fused_gemv_params(h, 0, l, emb, out, in_step), nb,
                      L.qkv.smem, s, h->pdl);
      break;
    case 1: {
      AttnParams p = k2_params(h, l);
      p.tl = (in_step && h->timeline) ? h->timeline + kTimelineSlots * (size_t)(l * 5 + 1) : nullptr;
      p.ahead = l2_ahead_of(h, 1, l);
      p.cluster = h->att_cluster;
      if (h->qpub) p.qout = h->qs[dec_handle::QS_O];
      e = launch_attn(h->d.head_dim, h->G, p, fused_att_grid(h), h->attn_smem, s, h->pdl);
      break;
    }
    case 2:
      e = launch_gemv(PRO_PLAIN, EPI_RESID, q4, fused_gemv_params(h, 2, l, emb, out, in_step), nb,
                      L.o.smem, s, h->pdl);
      break;
    case 3:
      e = launch_gemv(PRO_NORM, EPI_SWIGLU, q4, fused_gemv_params(h, 3, l, emb, out, in_step), nb,
                      L.gu.smem, s, h->pdl);
      break;
    case 4:
      e = launch_gemv(PRO_PLAIN, EPI_RESID, q4, fused_gemv_params(h, 4, l, emb, out, in_step), nb,
                      L.down.smem, s, h->pdl);
      break;
    default:
      return fail(h, DEC_ERR_ARG, "kernel id %d out of range", kernel);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  return DEC_OK;
}

int enqueue_unfused_layer(dec_handle* h, int l, const float* x_in, float* out, bool last,
                          cudaStream_t s) {
  const dec_model_desc& d = h->d;
  const LayerDev& L = h->layers[l];
  const int H = d.hidden, hd = d.head_dim, F = d.ffn, nq = d.n_q_heads, nkv = d.n_kv_heads;
  const bool q4 = d.weight_fmt == DEC_W_Q4B32;
  const int km = max_k(d);
  float* tap = h->tap ? h->tap + (size_t)l * H : nullptr;
#define TLD_U(call)                                        \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return cuda_fail(h, e_, #call); \
  } while (0)
  // q4: one quantisation per GEMV input vector (slot = q, o, gate/up, down)
  auto quant = [&](const float* z, int K, int slot) {
    int8_t* qt = h->qtap ? h->qtap + ((size_t)l * 4 + slot) * km : nullptr;
    float* st = h->qtap ? h->qstap + ((size_t)l * 4 + slot) * (km / 32) : nullptr;
    return unf::quantize(z, K, h->qbuf, h->dbuf, qt, st, s);
  };
  auto proj = [&](int m, int N, int K, const float* z, float* y) {
    return q4 ? unf::gemv_q4(L.q4n[m], L.q4s[m], N, K, h->qbuf, h->dbuf, y, s)
              : unf::gemv(L.mats[m], N, K, z, y, s);
  };
  TLD_U(unf::rms_scale(x_in, H, d.rms_eps, h->n1, s));
  TLD_U(unf::mul(h->n1, L.attn_norm, H, s));
  if (q4) TLD_U(quant(h->n1, H, 0));
  TLD_U(proj(0, nq * hd, H, h->n1, h->q));
  TLD_U(proj(1, nkv * hd, H, h->n1, h->k));
  TLD_U(proj(2, nkv * hd, H, h->n1, h->v));
  TLD_U(unf::rope(h->q, h->k, nq, nkv, hd, h->d_pos, h->rope, h->rope_inter ? 1 : 0, s));
  TLD_U(unf::kv_append(h->k, h->v, nkv, hd, d.max_ctx, h->d_pos, L.kc, L.vc, s));
  TLD_U(unf::attention(h->q, L.kc, L.vc, nq, nkv, hd, d.max_ctx, h->d_pos, h->o, s));
  if (q4) TLD_U(quant(h->o, nq * hd, 1));
  TLD_U(proj(3, H, nq * hd, h->o, h->y));
  TLD_U(unf::add(x_in, h->y, h->h1, nullptr, H, nullptr, s));
  TLD_U(unf::rms_scale(h->h1, H, d.rms_eps, h->n1, s));
  TLD_U(unf::mul(h->n1, L.ffn_norm, H, s));
  if (q4) TLD_U(quant(h->n1, H, 2));
  TLD_U(proj(4, F, H, h->n1, h->g));
  TLD_U(proj(5, F, H, h->n1, h->u));
  TLD_U(unf::swiglu(h->g, h->u, h->a, F, s));
  if (q4) TLD_U(quant(h->a, F, 3));
  TLD_U(proj(6, H, F, h->a, h->y));
  TLD_U(unf::add(h->h1, h->y, out, tap, H, last ? h->d_pos : nullptr, s));
#undef TLD_U
  return DEC_OK;
}
// one kernel per op; the q4 form adds one quantisation per GEMV input vector
constexpr int kUnfusedKernelsPerLayer = 17;
constexpr int kUnfusedKernelsPerLayerQ4 = 21;

// Parameters of the persistent per-token kernel for one step.
TokenParams token_params(const dec_handle* h, const float* emb, float* out) {
  TokenParams P{};
  const LayerDev& L0 = h->layers[0];
  P.layers = h->d_players;
  P.n_layers = h->d.n_layers;
  P.hidden = h->d.hidden;
  P.qkv = k1_params(h, 0, emb, false);
  P.o = k3_params(h, 0);
  P.gu = k4_params(h, 0);
  P.down = k5_params(h, 0, out, false);
  P.down.tap = nullptr;
  (void)L0;
  P.attn = k2_params(h, 0);
  P.att_grid = h->att_grid;
  P.emb = emb;
  P.out = out;
  P.X = h->X;
  P.tap = h->tap;
  P.pos = h->d_pos;
  P.bar = h->d_bar;
  P.err = h->d_err;
  P.nstages = h->p_nstages;
  P.slot_bytes = h->p_slot;
  P.qtap = h->qtap;
  P.qstap = h->qstap;
  P.km = max_k(h->d);
  P.dots = h->dot_tap;
  P.dot_layer = h->dot_layer;
  P.dot_kernel = h->dot_kernel;
  P.tl = h->timeline;
  return P;
}

int enqueue_layers(dec_handle* h, const float* emb, float* out, cudaStream_t s, bool capturing);

LmHeadParams lm_params(const dec_handle* h, const float* out) {
  LmHeadParams P{};
  P.g = gemv_base(h, h->lm);
  P.g.x = out;
  P.g.norm_w = h->lm_norm;
  P.g.out = h->logits_tap ? h->logits_tap : h->logits;
  P.key = h->lm_key;
  P.token_out = h->token_out;
  return P;
}

// The LM head and the greedy token after the stack's last layer (when the
// caller asked for tokens).
int enqueue_lm_head(dec_handle* h, const float* out, cudaStream_t s, bool capturing) {
  if (!h->token_out) return DEC_OK;
  cudaError_t e = launch_lm_head(lm_params(h, out), h->n_sm, h->lm.smem, s, h->pdl);
  if (e != cudaSuccess) return cuda_fail(h, e, "LM head launch");
  if (capturing) h->lm_node = last_captured_node(s);
  return DEC_OK;
}

// Queues one whole token.  Records the first and last kernel nodes when capturing.
int enqueue_step(dec_handle* h, const float* emb, float* out, cudaStream_t s, bool capturing) {
  const int rc = enqueue_layers(h, emb, out, s, capturing);
  if (rc) return rc;
  return enqueue_lm_head(h, out, s, capturing);
}

int enqueue_layers(dec_handle* h, const float* emb, float* out, cudaStream_t s, bool capturing) {
  const int Lc = h->d.n_layers;
  if (h->persistent) {
    cudaError_t e = launch_persistent(h->d.head_dim, h->G, h->d.weight_fmt == DEC_W_Q4B32,
                                      token_params(h, emb, out), h->n_sm, h->p_smem, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "persistent kernel launch");
    if (capturing) h->first_node = h->last_node = last_captured_node(s);
    return DEC_OK;
  }
  if (!h->fused) {
    for (int l = 0; l < Lc; ++l) {
      // the unfused chain ping-pongs the residual stream through X
      const float* xin = (l == 0) ? emb : h->X;
      float* xout = (l == Lc - 1) ? out : h->X;
      int rc = enqueue_unfused_layer(h, l, xin, xout, l == Lc - 1, s);
      if (rc) return rc;
    }
    return DEC_OK;
  }
  const int kpl = kernels_per_layer(h);
  for (int l = 0; l < Lc; ++l) {
    for (int k = 0; k < kpl; ++k) {
      int rc = enqueue_fused_kernel(h, k, l, emb, out, true, s);
      if (rc) return rc;
      if (capturing && l == 0 && k == 0) h->first_node = last_captured_node(s);
      if (capturing && l == Lc - 1 && k == kpl - 1) h->last_node = last_captured_node(s);
    }
  }
  return DEC_OK;
}

int capture(dec_handle* h, const float* emb, float* out) {
  drop_graph(h);
  if (!h->cap_stream) TLD_CUDA(h, cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
  TLD_CUDA(h, cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
  int rc = enqueue_step(h, emb, out, h->cap_stream, true);
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(h->cap_stream, &g);
  if (rc) {
    if (g) cudaGraphDestroy(g);
    return rc;
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamEndCapture");
  h->graph_g = g;
  TLD_CUDA(h, cudaGraphInstantiate(&h->exec, g, 0));
  if ((h->fused && (!h->first_node || !h->last_node)) || (h->token_out && !h->lm_node))
    return fail(h, DEC_ERR_CUDA, "could not locate the captured kernel nodes");
  h->cap_emb = emb;
  h->cap_out = out;
  return DEC_OK;
}

// The taps a captured launch of kernel k (0 QKV, 4 down) of layer l carries.
// Points the captured graph at new input / output buffers.
int patch_io_layers(dec_handle* h, const float* emb, float* out);

int patch_io(dec_handle* h, const float* emb, float* out) {
  if (!h->fused) return capture(h, emb, out);  // the unfused chain is only the ablation
  const float* old_out = h->cap_out;
  const int rc = patch_io_layers(h, emb, out);
  if (rc || !h->lm_node || out == old_out) return rc;
  // the LM head reads the stack's output
  LmHeadParams P = lm_params(h, out);
  void* args[] = {&P};
  cudaKernelNodeParams kp{};
  kp.func = const_cast<void*>(lm_head_kernel_ptr());
  kp.gridDim = dim3(h->n_sm);
  kp.blockDim = dim3(kThreads);
  kp.sharedMemBytes = (unsigned)h->lm.smem;
  kp.kernelParams = args;
  TLD_CUDA(h, cudaGraphExecKernelNodeSetParams(h->exec, h->lm_node, &kp));
  return DEC_OK;
}

int patch_io_layers(dec_handle* h, const float* emb, float* out) {
  if (h->persistent) {
    if (emb == h->cap_emb && out == h->cap_out) return DEC_OK;
    TokenParams P = token_params(h, emb, out);
    void* args[] = {&P};
    cudaKernelNodeParams kp{};
    kp.func = const_cast<void*>(
        persistent_kernel_ptr(h->d.head_dim, h->G, h->d.weight_fmt == DEC_W_Q4B32));
    kp.gridDim = dim3(h->n_sm);
    kp.blockDim = dim3(kThreads);
    kp.sharedMemBytes = (unsigned)h->p_smem;
    kp.kernelParams = args;
    TLD_CUDA(h, cudaGraphExecKernelNodeSetParams(h->exec, h->first_node, &kp));
    h->cap_emb = emb;
    h->cap_out = out;
    return DEC_OK;
  }
  if (emb != h->cap_emb) {
    GemvParams p = fused_gemv_params(h, 0, 0, emb, out, true);
    void* args[] = {&p};
    cudaKernelNodeParams kp{};
    kp.func = const_cast<void*>(gemv_kernel_ptr(PRO_NORM, EPI_QKV, h->d.weight_fmt == DEC_W_Q4B32));
    kp.gridDim = dim3(h->n_sm);
    kp.blockDim = dim3(kThreads);
    kp.sharedMemBytes = (unsigned)h->layers[0].qkv.smem;
    kp.kernelParams = args;
    TLD_CUDA(h, cudaGraphExecKernelNodeSetParams(h->exec, h->first_node, &kp));
    h->cap_emb = emb;
  }
  if (out != h->cap_out && (h->three || h->four)) {
    const int l = h->d.n_layers - 1;
    FfnParams p = ffn_params(h, l, emb, out, true);
    void* args[] = {&p};
    cudaKernelNodeParams kp{};
    kp.func = const_cast<void*>(ffn_kernel_ptr(h->d.weight_fmt == DEC_W_Q4B32));
    kp.gridDim = dim3(h->n_sm);
    kp.blockDim = dim3(kThreads);
    kp.sharedMemBytes = (unsigned)h->ffn_smem;
    kp.kernelParams = args;
    TLD_CUDA(h, cudaGraphExecKernelNodeSetParams(h->exec, h->last_node, &kp));
    h->cap_out = out;
  }
  if (out != h->cap_out) {
    const int l = h->d.n_layers - 1;
    GemvParams p = fused_gemv_params(h, 4, l, emb, out, true);
    void* args[] = {&p};
    cudaKernelNodeParams kp{};
    kp.func = const_cast<void*>(gemv_kernel_ptr(PRO_PLAIN, EPI_RESID, h->d.weight_fmt == DEC_W_Q4B32));
    kp.gridDim = dim3(h->n_sm);
    kp.blockDim = dim3(kThreads);
    kp.sharedMemBytes = (unsigned)h->layers[l].down.smem;
    kp.kernelParams = args;
    TLD_CUDA(h, cudaGraphExecKernelNodeSetParams(h->exec, h->last_node, &kp));
    h->cap_out = out;
  }
  return DEC_OK;
}

int set_device_pos(dec_handle* h, int pos) {
  TLD_CUDA(h, cudaMemcpy(h->d_pos, &pos, sizeof(int), cudaMemcpyHostToDevice));
  // the persistent kernel's barrier counters alternate by position parity:
  // after a jump of the position both start from zero
  if (h->d_bar) TLD_CUDA(h, cudaMemset(h->d_bar, 0, 2 * sizeof(int)));
  if (h->d_fbar) TLD_CUDA(h, cudaMemset(h->d_fbar, 0, 4 * sizeof(int) * (size_t)h->d.n_layers));
  return DEC_OK;
}

}  // namespace

// ---- C ABI ----------------------------------------------------------------------

extern "C" {

int dec_create(const dec_model_desc* desc, dec_handle** out) {
  if (!out) return fail(nullptr, DEC_ERR_ARG, "out is NULL");
  *out = nullptr;
  if (!desc) return fail(nullptr, DEC_ERR_ARG, "desc is NULL");
  const dec_model_desc d = *desc;
  if (d.n_layers < 1 || d.hidden < 1 || d.n_q_heads < 1 || d.n_kv_heads < 1 || d.ffn < 1 ||
      d.max_ctx < 1 || !(d.rms_eps >= 0.f) || !(d.rope_theta > 0.f))
    return fail(nullptr, DEC_ERR_ARG, "non-positive size or bad eps/theta in the model desc");
  if (d.head_dim != 64 && d.head_dim != 128)
    return fail(nullptr, DEC_ERR_SHAPE, "head_dim %d unsupported (64 or 128)", d.head_dim);
  if (d.n_q_heads % d.n_kv_heads)
    return fail(nullptr, DEC_ERR_SHAPE, "n_q_heads %% n_kv_heads != 0");
  const int G = d.n_q_heads / d.n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(nullptr, DEC_ERR_SHAPE, "GQA group %d unsupported (1, 2, 4 or 8)", G);
  if (d.hidden % 8 || d.ffn % 8)
    return fail(nullptr, DEC_ERR_SHAPE, "hidden and ffn must be multiples of 8");
  if (d.max_ctx > 65536) return fail(nullptr, DEC_ERR_SHAPE, "max_ctx > 65536");
  if (d.weight_fmt != DEC_W_BF16 && d.weight_fmt != DEC_W_Q4B32)
    return fail(nullptr, DEC_ERR_ARG, "unknown weight_fmt %d", d.weight_fmt);
  if (d.weight_fmt == DEC_W_Q4B32 &&
      (d.hidden % 64 || d.ffn % 64 || (d.n_q_heads * d.head_dim) % 64))
    return fail(nullptr, DEC_ERR_SHAPE, "int4 weights need hidden, ffn and heads*head_dim multiples of 64");
  if (d.flags & ~(DEC_PLAN_UNFUSED | DEC_NO_GRAPH | DEC_NO_PDL | DEC_PLAN_PERSISTENT | DEC_NO_L2_AHEAD |
                  DEC_ATTN_GLOBAL_MERGE | DEC_PLAN_THREE | DEC_DEBUG_GUARDS | DEC_ROPE_INTERLEAVED |
                  DEC_PAGED_KV | DEC_PLAN_FOUR | DEC_Q4_PUBLISH | DEC_FUSE_ATTN_OPROJ))
    return fail(nullptr, DEC_ERR_ARG, "unknown flags 0x%x", d.flags);

  dec_handle* h = new (std::nothrow) dec_handle();
  if (!h) return fail(nullptr, DEC_ERR_OOM, "host allocation failed");
  h->d = d;
  h->G = G;
  h->fused = !(d.flags & DEC_PLAN_UNFUSED);
  h->graph = !(d.flags & DEC_NO_GRAPH);
  h->pdl = !(d.flags & DEC_NO_PDL);
  h->l2_ahead = !(d.flags & DEC_NO_L2_AHEAD);
  h->cluster_attn = !(d.flags & DEC_ATTN_GLOBAL_MERGE);
  h->persistent = h->fused && (d.flags & DEC_PLAN_PERSISTENT);
  h->three = h->fused && !h->persistent && (d.flags & DEC_PLAN_THREE);
  h->four = h->fused && !h->persistent && !h->three && (d.flags & DEC_PLAN_FOUR);
  h->headproj = h->fused && !h->persistent && !h->three && (d.flags & DEC_FUSE_ATTN_OPROJ);
  h->qpub = h->fused && !h->persistent && !h->three && !h->headproj &&
            d.weight_fmt == DEC_W_Q4B32 && (d.flags & DEC_Q4_PUBLISH);
  h->guards = (d.flags & DEC_DEBUG_GUARDS) != 0;
  h->rope_inter = (d.flags & DEC_ROPE_INTERLEAVED) != 0;
  h->paged = (d.flags & DEC_PAGED_KV) != 0;
  if (h->paged && !h->fused) {
    delete h;
    return fail(nullptr, DEC_ERR_SHAPE, "the paged KV cache needs a fused plan");
  }
  h->page_rows = kAttnStageBytes / 4 / d.head_dim;  // one attention chunk
  h->n_pages = (d.max_ctx + h->page_rows - 1) / h->page_rows;
  if (h->three) h->cluster_attn = false;  // its attention phase is a flat grid
  if (h->headproj && !h->cluster_attn) {
    delete h;
    return fail(nullptr, DEC_ERR_SHAPE, "the fused attention + o-projection needs the cluster attention");
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = set_smem_limits();
  if (e != cudaSuccess) {
    g_create_error = std::string("CUDA device query: ") + cudaGetErrorString(e);
    delete h;
    return DEC_ERR_CUDA;
  }
  const int H = d.hidden, hd = d.head_dim, F = d.ffn, nq = d.n_q_heads, nkv = d.n_kv_heads;
  // attention grid: at most kMaxSplits - 1 CTAs per KV head, so a head is never
  // split over more than kMaxSplits CTAs
  h->att_grid = h->n_sm < (kMaxSplits - 1) * nkv ? h->n_sm : (kMaxSplits - 1) * nkv;
  int rc = DEC_OK;
  auto A = [&](auto** p, size_t bytes, int64_t* acct) {
    if (rc == DEC_OK) rc = dev_alloc(h, p, bytes, acct);
  };
  h->layers.resize(d.n_layers);
  for (int l = 0; l < d.n_layers; ++l) {
    LayerDev& L = h->layers[l];
    A(&L.attn_norm, 2 * (size_t)H, &h->weight_bytes);
    A(&L.ffn_norm, 2 * (size_t)H, &h->weight_bytes);
    if (h->fused) {
      const bool q4 = d.weight_fmt == DEC_W_Q4B32;
      plan_tiled(L.qkv, (nq + 2 * nkv) * hd, H, h->n_sm, q4);
      plan_tiled(L.o, H, nq * hd, h->n_sm, q4);
      plan_tiled(L.gu, 2 * F, H, h->n_sm, q4);
      plan_tiled(L.down, H, F, h->n_sm, q4);
      for (Tiled* t : {&L.qkv, &L.o, &L.gu, &L.down}) A(&t->w, t->bytes, &h->weight_bytes);
    } else {
      for (int m = 0; m < kNumMats; ++m) {
        int N, K;
        mat_shape(d, DEC_T_WQ + (m < 4 ? m : m + 1), &N, &K);
        if (d.weight_fmt == DEC_W_Q4B32) {
          A(&L.q4n[m], (size_t)N * K / 2, &h->weight_bytes);
          A(&L.q4s[m], (size_t)N * (K / 32) * 2, &h->weight_bytes);
        } else {
          A(&L.mats[m], 2 * (size_t)N * K, &h->weight_bytes);
        }
      }
    }
    const size_t kv_elems = h->paged ? (size_t)h->n_pages * nkv * h->page_rows * hd
                                     : (size_t)nkv * d.max_ctx * hd;
    A(&L.kc, 2 * kv_elems, &h->kv_bytes);
    A(&L.vc, 2 * kv_elems, &h->kv_bytes);
  }
  const int km = max_k(d);
  A(&h->X, 4 * (size_t)H, &h->ws_bytes);
  A(&h->h1, 4 * (size_t)H, &h->ws_bytes);
  A(&h->q, 4 * (size_t)nq * hd, &h->ws_bytes);
  A(&h->o, 4 * (size_t)nq * hd, &h->ws_bytes);
  A(&h->a, 4 * (size_t)F, &h->ws_bytes);
  A(&h->n1, 4 * (size_t)H, &h->ws_bytes);
  A(&h->k, 4 * (size_t)nkv * hd, &h->ws_bytes);
  A(&h->v, 4 * (size_t)nkv * hd, &h->ws_bytes);
  A(&h->g, 4 * (size_t)F, &h->ws_bytes);
  A(&h->u, 4 * (size_t)F, &h->ws_bytes);
  A(&h->y, 4 * (size_t)km, &h->ws_bytes);
  A(&h->qbuf, (size_t)km, &h->ws_bytes);
  A(&h->dbuf, 4 * (size_t)(km / 32 + 1), &h->ws_bytes);
  A(&h->apart, 4 * (size_t)h->att_grid * 2 * G * (hd + 4), &h->ws_bytes);
  A(&h->acount, 4 * (size_t)nkv, &h->ws_bytes);
  if (h->persistent) {
    A(&h->d_players, sizeof(PLayer) * (size_t)d.n_layers, &h->ws_bytes);
    A(&h->d_bar, 16, &h->ws_bytes);
  }
  if (h->three || h->four) A(&h->d_fbar, 4 * sizeof(int) * (size_t)d.n_layers, &h->ws_bytes);
  if (h->paged) A(&h->d_pages, sizeof(int) * (size_t)h->n_pages, &h->ws_bytes);
  if (h->headproj) {
    A(&h->hp_part, 4 * (size_t)nkv * H, &h->ws_bytes);
    A(&h->hp_cnt, sizeof(int) * (size_t)kMaxCluster, &h->ws_bytes);
    const bool q4 = d.weight_fmt == DEC_W_Q4B32;
    h->hp_geo = tile_geom(G * hd, q4);
    h->hp_group_bytes = (int64_t)(H / kTileR) * h->hp_geo.rb_bytes;
  }
  // the GEMV reading a published RMSNorm input stages the producers' per-CTA
  // sums of squares in its K-float input buffer
  if (h->qpub && H < h->n_sm) h->qpub = false;
  if (h->qpub) {
    const int qk[4] = {H, nq * hd, H, F};
    for (int i = 0; i < 4; ++i) {
      QVec& q = h->qs[i];
      q.K = qk[i];
      A(&q.codes, (size_t)q.K, &h->ws_bytes);
      A(&q.scale, 4 * (size_t)(q.K / 32), &h->ws_bytes);
      A(&q.sum, 4 * (size_t)(q.K / 32), &h->ws_bytes);
      if (i != dec_handle::QS_O) A(&q.cnt, 4 * (size_t)(q.K / 32), &h->ws_bytes);  // o: whole blocks
      if (i == dec_handle::QS_N1 || i == dec_handle::QS_N2) {  // RMSNorm inputs
        q.n_part = h->n_sm;
        A(&q.part, 4 * (size_t)h->n_sm, &h->ws_bytes);
      }
    }
  }
  A(&h->d_pos, 16, &h->ws_bytes);
  A(&h->d_err, 16, &h->ws_bytes);
  A(&h->rope, sizeof(float2) * (size_t)d.max_ctx * (hd / 2), &h->ws_bytes);
  if (rc) {
    dec_destroy(h);
    g_create_error = "device allocation failed";
    return rc;
  }
  // zero the flags / position / partials; fill the RoPE table in double
  e = cudaMemset(h->d_pos, 0, 16);
  if (e == cudaSuccess) e = cudaMemset(h->apart, 0, 4 * (size_t)h->att_grid * 2 * G * (hd + 4));
  if (e == cudaSuccess) e = cudaMemset(h->acount, 0, 4 * (size_t)nkv);
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, 16);
  if (e == cudaSuccess) {
    std::vector<float2> tab((size_t)d.max_ctx * (hd / 2));
    for (int p = 0; p < d.max_ctx; ++p)
      for (int i = 0; i < hd / 2; ++i) {
        const double ang = (double)p * std::pow((double)d.rope_theta, -2.0 * i / hd);
        tab[(size_t)p * (hd / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    e = cudaMemcpy(h->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess && h->d_fbar) e = cudaMemset(h->d_fbar, 0, 4 * sizeof(int) * (size_t)d.n_layers);
  for (int i = 0; i < 4 && e == cudaSuccess; ++i)
    if (h->qs[i].cnt) e = cudaMemset(h->qs[i].cnt, 0, 4 * (size_t)(h->qs[i].K / 32));
  if (e == cudaSuccess && h->hp_cnt) e = cudaMemset(h->hp_cnt, 0, sizeof(int) * (size_t)kMaxCluster);
  if (e == cudaSuccess && h->paged) {  // identity page table until the caller sets one
    h->h_pages.resize(h->n_pages);
    for (int c = 0; c < h->n_pages; ++c) h->h_pages[c] = c;
    e = cudaMemcpy(h->d_pages, h->h_pages.data(), sizeof(int) * h->h_pages.size(),
                   cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess && h->persistent) {
    std::vector<PLayer> pl(d.n_layers);
    for (int l = 0; l < d.n_layers; ++l) {
      const LayerDev& L = h->layers[l];
      pl[l] = PLayer{L.qkv.w, L.o.w, L.gu.w, L.down.w, L.attn_norm, L.ffn_norm, L.kc, L.vc};
    }
    e = cudaMemcpy(h->d_players, pl.data(), sizeof(PLayer) * pl.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(h->d_bar, 0, 16);
  }
  if (e != cudaSuccess) {
    g_create_error = std::string("initialising device buffers: ") + cudaGetErrorString(e);
    dec_destroy(h);
    return DEC_ERR_CUDA;
  }
  {
    const bool cl = h->fused && !h->persistent && h->cluster_attn;
    const size_t fixed = attn_smem_bytes(hd, G, 0, cl);
    int ns = (int)(((size_t)kSmemBudget > fixed ? kSmemBudget - fixed : 0) / kAttnStageBytes);
    h->attn_nstages = ns < 2 ? 2 : (ns > 6 ? 6 : ns);
    h->attn_smem = attn_smem_bytes(hd, G, h->attn_nstages, cl);
  }
  if (h->three || h->four) {
    // ring slots hold an attention chunk or a GEMV stage; as many as the budget
    // leaves next to the larger of the two phases' work areas
    const bool q4 = d.weight_fmt == DEC_W_Q4B32;
    const int gstage = q4 ? kStageBytesQ4 : kStageBytes;
    const LayerDev& L0 = h->layers[0];
    auto stages = [](size_t fixed, int slot) {
      int ns = (int)(((size_t)kSmemBudget > fixed ? kSmemBudget - fixed : 0) / (slot + 16));
      return ns < 2 ? 2 : (ns > 8 ? 8 : ns);
    };
    h->ao_slot = gstage > kAttnStageBytes ? gstage : kAttnStageBytes;
    h->ao_nstages = stages(attn_oproj_smem_bytes(hd, G, nq * hd, L0.o.max_rb_local, q4, 0, 0),
                           h->ao_slot);
    h->ao_smem = attn_oproj_smem_bytes(hd, G, nq * hd, L0.o.max_rb_local, q4, h->ao_nstages,
                                       h->ao_slot);
    h->ffn_slot = gstage;
    h->ffn_nstages = stages(ffn_smem_bytes(H, L0.gu.max_rb_local, F, L0.down.max_rb_local, q4, 0, 0),
                            h->ffn_slot);
    h->ffn_smem = ffn_smem_bytes(H, L0.gu.max_rb_local, F, L0.down.max_rb_local, q4,
                                 h->ffn_nstages, h->ffn_slot);
    // The in-kernel grid barrier needs every CTA of the grid (one per SM)
    // resident at once: refuse a plan whose CTA does not fit on an SM.
    struct {
      const void* fn;
      size_t smem;
    } two_phase[2] = {{ffn_kernel_ptr(q4), h->ffn_smem},
                      {h->three ? attn_oproj_kernel_ptr(hd, G, q4) : nullptr, h->ao_smem}};
    for (const auto& k : two_phase) {
      if (!k.fn) continue;
      int per_sm = 0;
      e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, kThreads, k.smem);
      if (e != cudaSuccess || per_sm < 1) {
        g_create_error = std::string("two-phase kernel cannot be resident: ") +
                         (e != cudaSuccess ? cudaGetErrorString(e) : "no room on an SM");
        dec_destroy(h);
        return e != cudaSuccess ? DEC_ERR_CUDA : DEC_ERR_SHAPE;
      }
    }
  }
  if (h->fused && !h->persistent && h->cluster_attn) {
    // one cluster per KV head, as many CTAs per head as the SMs allow with every
    // cluster resident at once (one wave)
    int C = h->n_sm / nkv;
    if (C > kMaxCluster) C = kMaxCluster;
    if (C < 1) C = 1;
    const bool q4 = d.weight_fmt == DEC_W_Q4B32;
    const void* fn = h->headproj ? attn_headproj_kernel_ptr(hd, G, q4) : attn_kernel_ptr(hd, G, true);
    auto hp_size = [&](int c) {  // ring stages and shared memory of the fused kernel at cluster size c
      const int quads = (H / kTileR + c - 1) / c;
      const size_t fixed = attn_headproj_smem_bytes(hd, G, q4, 0, quads, nkv);
      int ns = (int)(((size_t)kSmemBudget > fixed ? kSmemBudget - fixed : 0) / (kAttnStageBytes + 16));
      ns = ns < 2 ? 2 : (ns > 6 ? 6 : ns);
      h->hp_nstages = ns;
      h->hp_smem = attn_headproj_smem_bytes(hd, G, q4, ns, quads, nkv);
    };
    for (; C > 1; --C) {
      if (h->headproj) hp_size(C);
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(nkv * C);
      cfg.blockDim = dim3(h->headproj ? kThreads : (attn_consumer_warps(hd, G, true) + 1) * 32);
      cfg.dynamicSmemBytes = h->headproj ? h->hp_smem : h->attn_smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = C;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int active = 0;
      if (cudaOccupancyMaxActiveClusters(&active, fn, &cfg) == cudaSuccess && active >= nkv) break;
      cudaGetLastError();  // a size the device refuses is not an error of the handle
    }
    if (h->headproj) hp_size(C);
    h->att_cluster = C;
  }
  if (h->persistent) {
    // one ring for every phase: slots as large as the largest stage; the work
    // area is the largest phase's; all of it within one CTA per SM
    const bool q4 = d.weight_fmt == DEC_W_Q4B32;
    h->p_slot = q4 ? kStageBytesQ4 : kStageBytes;
    if (kAttnStageBytes > h->p_slot) h->p_slot = kAttnStageBytes;
    h->p_nstages = 1;  // placeholder for the work-size query
    const size_t work = persistent_work_bytes(token_params(h, nullptr, nullptr), hd, G, q4);
    int ns = (int)(((size_t)kSmemBudget > work ? kSmemBudget - work : 0) / (h->p_slot + 16));
    ns = ns < 2 ? 2 : (ns > 8 ? 8 : ns);
    h->p_nstages = ns;
    h->p_smem = (size_t)ns * h->p_slot + 16 * (size_t)ns + work;
    int per_sm = 0;
    const void* fn = persistent_kernel_ptr(hd, G, q4);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->p_smem);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, h->p_smem);
    if (e != cudaSuccess || per_sm < 1) {
      g_create_error = std::string("persistent kernel cannot be resident: ") +
                       (e != cudaSuccess ? cudaGetErrorString(e) : "no room on an SM");
      dec_destroy(h);
      return e != cudaSuccess ? DEC_ERR_CUDA : DEC_ERR_SHAPE;
    }
  }
  *out = h;
  return DEC_OK;
}

int dec_load_weights(dec_handle* h, int layer, int tensor, const void* src, size_t bytes) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (!src) return fail(h, DEC_ERR_ARG, "src is NULL");
  const dec_model_desc& d = h->d;
  if (layer < 0 || layer >= d.n_layers) return fail(h, DEC_ERR_ARG, "layer %d out of range", layer);
  LayerDev& L = h->layers[layer];
  if (tensor == DEC_T_ATTN_NORM || tensor == DEC_T_FFN_NORM) {
    if (bytes != 2 * (size_t)d.hidden)
      return fail(h, DEC_ERR_ARG, "norm vector: %zu bytes, expected %zu", bytes, 2 * (size_t)d.hidden);
    TLD_CUDA(h, cudaMemcpy(tensor == DEC_T_ATTN_NORM ? L.attn_norm : L.ffn_norm, src, bytes,
                           cudaMemcpyDefault));
    L.loaded |= 1u << tensor;
    return DEC_OK;
  }
  const bool q4 = d.weight_fmt == DEC_W_Q4B32;
  const bool scales = q4 && tensor >= DEC_T_SCALES;
  const int mt = scales ? tensor - DEC_T_SCALES : tensor;
  int N, K;
  mat_shape(d, mt, &N, &K);
  if (N == 0) return fail(h, DEC_ERR_ARG, "tensor id %d invalid for this weight format", tensor);
  const size_t want = !q4 ? 2 * (size_t)N * K : scales ? (size_t)N * (K / 32) * 2 : (size_t)N * K / 2;
  if (bytes != want) return fail(h, DEC_ERR_ARG, "tensor %d: %zu bytes, expected %zu", tensor, bytes, want);
  if (!h->fused) {
    const int m = mat_index(mt);
    void* dst = !q4 ? (void*)L.mats[m] : scales ? (void*)L.q4s[m] : (void*)L.q4n[m];
    TLD_CUDA(h, cudaMemcpy(dst, src, bytes, cudaMemcpyDefault));
    L.loaded |= 1u << tensor;
    return DEC_OK;
  }
  if (h->staging_bytes < want) {
    if (h->staging) {
      uint8_t* user = reinterpret_cast<uint8_t*>(h->staging);
      void* base = h->guards ? user - kGuardBytes : user;
      cudaFree(base);
      for (auto& p : h->allocs)
        if (p == base) p = nullptr;
      for (auto& g : h->guard_list)
        if (g.user == user) g.bytes = 0;  // gone: nothing to check
    }
    h->staging = nullptr;
    h->staging_bytes = 0;
    int rc = dev_alloc(h, &h->staging, want, nullptr);
    if (rc) return rc;
    h->staging_bytes = want;
  }
  TLD_CUDA(h, cudaMemcpy(h->staging, src, bytes, cudaMemcpyDefault));
  const int hd = d.head_dim;
  // destination matrix, first tiled row and row map of each tensor
  uint8_t* dst = nullptr;
  int row0 = 0, kind = 0;
  switch (mt) {
    // q/k rows: a RoPE pair's two rows adjacent (pairs (i, i+hd/2) interleaved;
    // pairs (2i, 2i+1) already are)
    case DEC_T_WQ: dst = L.qkv.w; row0 = 0; kind = h->rope_inter ? 0 : 1; break;
    case DEC_T_WK: dst = L.qkv.w; row0 = d.n_q_heads * hd; kind = h->rope_inter ? 0 : 1; break;
    case DEC_T_WV: dst = L.qkv.w; row0 = (d.n_q_heads + d.n_kv_heads) * hd; kind = 0; break;
    case DEC_T_WO: dst = L.o.w; row0 = 0; kind = 0; break;
    case DEC_T_WGATE: dst = L.gu.w; row0 = 0; kind = 2; break;
    case DEC_T_WUP: dst = L.gu.w; row0 = 1; kind = 2; break;
    default: dst = L.down.w; row0 = 0; kind = 0; break;
  }
  cudaError_t e;
  if (mt == DEC_T_WO && h->headproj)  // stored per KV-head group (columns of G heads)
    e = launch_repack_groups(h->staging, scales, q4, N, K, h->G * hd, dst, h->hp_group_bytes, 0);
  else if (!q4)
    e = launch_repack_bf16(h->staging, N, K, dst, row0, kind, hd, 0);
  else if (scales)
    e = launch_repack_q4(nullptr, h->staging, N, K, dst, row0, kind, hd, 0);
  else
    e = launch_repack_q4(reinterpret_cast<const uint8_t*>(h->staging), nullptr, N, K, dst, row0,
                         kind, hd, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "weight repack");
  L.loaded |= 1u << tensor;
  return DEC_OK;
}

int dec_load_kv(dec_handle* h, int layer, const void* k_bf16, const void* v_bf16, int n_pos) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  const dec_model_desc& d = h->d;
  if (layer < 0 || layer >= d.n_layers) return fail(h, DEC_ERR_ARG, "layer %d out of range", layer);
  if (n_pos < 0) return fail(h, DEC_ERR_ARG, "n_pos < 0");
  if (n_pos >= d.max_ctx) return fail(h, DEC_ERR_CTX, "n_pos %d leaves no room (max_ctx %d)", n_pos, d.max_ctx);
  if (n_pos > 0 && (!k_bf16 || !v_bf16)) return fail(h, DEC_ERR_ARG, "k or v is NULL");
  TLD_CUDA(h, cudaDeviceSynchronize());
  LayerDev& L = h->layers[layer];
  if (n_pos > 0) {
    const int hd = d.head_dim;
    int rc = for_kv_runs(h, 0, n_pos, [&](int64_t off, int rows, int64_t src_row) -> int {
      const size_t n = 2 * (size_t)rows * hd;
      const size_t so = 2 * (size_t)src_row * hd;
      TLD_CUDA(h, cudaMemcpy(L.kc + off, static_cast<const uint8_t*>(k_bf16) + so, n, cudaMemcpyDefault));
      TLD_CUDA(h, cudaMemcpy(L.vc + off, static_cast<const uint8_t*>(v_bf16) + so, n, cudaMemcpyDefault));
      return DEC_OK;
    });
    if (rc) return rc;
  }
  if (h->guards && n_pos < d.max_ctx) {  // rows past the new length hold poison again
    int rc = for_kv_runs(h, n_pos, d.max_ctx, [&](int64_t off, int rows, int64_t) -> int {
      for (uint16_t* c : {L.kc, L.vc})
        TLD_CUDA(h, cudaMemset(c + off, 0xFF, 2 * (size_t)rows * d.head_dim));
      return DEC_OK;
    });
    if (rc) return rc;
  }
  L.kv_len = n_pos;
  h->kv_len = n_pos;
  return set_device_pos(h, n_pos);
}

int dec_load_lm_head(dec_handle* h, const void* final_norm_bf16, const void* w_bf16, int vocab) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (!final_norm_bf16 || !w_bf16) return fail(h, DEC_ERR_ARG, "final norm or LM head weights NULL");
  if (vocab < kTileR || vocab % kTileR)
    return fail(h, DEC_ERR_SHAPE, "vocab %d: a positive multiple of %d", vocab, kTileR);
  if (h->lm_loaded && vocab != h->vocab)
    return fail(h, DEC_ERR_ARG, "vocab %d differs from the loaded %d", vocab, h->vocab);
  const int H = h->d.hidden;
  if (!h->lm_loaded) {
    plan_tiled(h->lm, vocab, H, h->n_sm, false);
    int rc = dev_alloc(h, &h->lm.w, h->lm.bytes, &h->weight_bytes);
    if (!rc) rc = dev_alloc(h, &h->lm_norm, 2 * (size_t)H, &h->weight_bytes);
    if (!rc) rc = dev_alloc(h, &h->logits, 4 * (size_t)vocab, &h->ws_bytes);
    if (!rc) rc = dev_alloc(h, &h->lm_key, 16, &h->ws_bytes);
    if (rc) return rc;
    TLD_CUDA(h, cudaMemset(h->lm_key, 0, 16));
    h->vocab = vocab;
  }
  const size_t want = 2 * (size_t)vocab * H;
  if (h->staging_bytes < want) {
    if (h->staging) {
      uint8_t* user = reinterpret_cast<uint8_t*>(h->staging);
      void* base = h->guards ? user - kGuardBytes : user;
      cudaFree(base);
      for (auto& p : h->allocs)
        if (p == base) p = nullptr;
      for (auto& g : h->guard_list)
        if (g.user == user) g.bytes = 0;
    }
    h->staging = nullptr;
    h->staging_bytes = 0;
    int rc = dev_alloc(h, &h->staging, want, nullptr);
    if (rc) return rc;
    h->staging_bytes = want;
  }
  TLD_CUDA(h, cudaMemcpy(h->lm_norm, final_norm_bf16, 2 * (size_t)H, cudaMemcpyDefault));
  TLD_CUDA(h, cudaMemcpy(h->staging, w_bf16, want, cudaMemcpyDefault));
  cudaError_t e = launch_repack_bf16(h->staging, vocab, H, h->lm.w, 0, 0, h->d.head_dim, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(h, e, "LM head repack");
  h->lm_loaded = true;
  drop_graph(h);
  return DEC_OK;
}

int dec_set_token_out(dec_handle* h, int32_t* token_out, float* logits_tap) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (token_out && !h->lm_loaded) return fail(h, DEC_ERR_STATE, "no LM head loaded (dec_load_lm_head)");
  if (logits_tap && !token_out) return fail(h, DEC_ERR_ARG, "a logits tap needs token_out");
  h->token_out = token_out;
  h->logits_tap = logits_tap;
  drop_graph(h);
  return DEC_OK;
}

int dec_set_page_table(dec_handle* h, const int32_t* pages, int n) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (!h->paged) return fail(h, DEC_ERR_STATE, "the handle was created without DEC_PAGED_KV");
  if (!pages || n != h->n_pages)
    return fail(h, DEC_ERR_ARG, "the page table has %d entries, expected %d", n, h->n_pages);
  std::vector<int> t(n), seen(n, 0);
  TLD_CUDA(h, cudaMemcpy(t.data(), pages, sizeof(int) * (size_t)n, cudaMemcpyDefault));
  for (int c = 0; c < n; ++c) {
    if (t[c] < 0 || t[c] >= n || seen[t[c]]++)
      return fail(h, DEC_ERR_ARG, "page table entry %d (%d) out of range or repeated", c, t[c]);
  }
  // the rows already in the cache move with their pages
  TLD_CUDA(h, cudaDeviceSynchronize());
  const dec_model_desc& d = h->d;
  const size_t page_elems = (size_t)d.n_kv_heads * h->page_rows * d.head_dim;
  const size_t page_bytes = 2 * page_elems;
  std::vector<uint8_t> tmp(page_bytes * (size_t)n);
  for (LayerDev& L : h->layers)
    for (uint16_t* c : {L.kc, L.vc}) {
      TLD_CUDA(h, cudaMemcpy(tmp.data(), c, tmp.size(), cudaMemcpyDeviceToHost));
      for (int ch = 0; ch < n; ++ch)
        TLD_CUDA(h, cudaMemcpy(c + (size_t)t[ch] * page_elems, tmp.data() + (size_t)h->h_pages[ch] * page_bytes,
                               page_bytes, cudaMemcpyHostToDevice));
    }
  h->h_pages = t;
  TLD_CUDA(h, cudaMemcpy(h->d_pages, t.data(), sizeof(int) * (size_t)n, cudaMemcpyHostToDevice));
  return DEC_OK;
}

int dec_read_kv(dec_handle* h, int layer, void* k_bf16, void* v_bf16, int first_pos, int n_pos) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  const dec_model_desc& d = h->d;
  if (layer < 0 || layer >= d.n_layers) return fail(h, DEC_ERR_ARG, "layer %d out of range", layer);
  if (first_pos < 0 || n_pos < 0 || first_pos + n_pos > d.max_ctx)
    return fail(h, DEC_ERR_ARG, "rows [%d, %d) outside the cache (max_ctx %d)", first_pos,
                first_pos + n_pos, d.max_ctx);
  if (n_pos > 0 && (!k_bf16 || !v_bf16)) return fail(h, DEC_ERR_ARG, "k or v is NULL");
  TLD_CUDA(h, cudaDeviceSynchronize());
  if (n_pos == 0) return DEC_OK;
  const LayerDev& L = h->layers[layer];
  return for_kv_runs(h, first_pos, first_pos + n_pos, [&](int64_t off, int rows, int64_t dst_row) -> int {
    const size_t n = 2 * (size_t)rows * d.head_dim;
    const size_t so = 2 * (size_t)dst_row * d.head_dim;
    TLD_CUDA(h, cudaMemcpy(static_cast<uint8_t*>(k_bf16) + so, L.kc + off, n, cudaMemcpyDefault));
    TLD_CUDA(h, cudaMemcpy(static_cast<uint8_t*>(v_bf16) + so, L.vc + off, n, cudaMemcpyDefault));
    return DEC_OK;
  });
}

int dec_truncate_kv(dec_handle* h, int n_pos) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  for (const LayerDev& L : h->layers)
    if (n_pos < 0 || n_pos > L.kv_len)
      return fail(h, DEC_ERR_POS, "truncate to %d beyond a layer's KV length %d", n_pos, L.kv_len);
  TLD_CUDA(h, cudaDeviceSynchronize());
  const dec_model_desc& d = h->d;
  for (LayerDev& L : h->layers) {
    if (h->guards && n_pos < d.max_ctx) {  // rows past the new length hold poison again
      int rc = for_kv_runs(h, n_pos, d.max_ctx, [&](int64_t off, int rows, int64_t) -> int {
        for (uint16_t* c : {L.kc, L.vc})
          TLD_CUDA(h, cudaMemset(c + off, 0xFF, 2 * (size_t)rows * d.head_dim));
        return DEC_OK;
      });
      if (rc) return rc;
    }
    L.kv_len = n_pos;
  }
  h->kv_len = n_pos;
  return set_device_pos(h, n_pos);
}

int dec_step(dec_handle* h, const float* emb, int pos, float* out, dec_stream_t stream) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (!emb || !out) return fail(h, DEC_ERR_ARG, "token_embedding or out_hidden is NULL");
  const uint32_t need = required_mask(h->d);
  for (int l = 0; l < h->d.n_layers; ++l) {
    const LayerDev& L = h->layers[l];
    if ((L.loaded & need) != need)
      return fail(h, DEC_ERR_STATE, "layer %d: weights not all loaded (mask 0x%x of 0x%x)", l,
                  L.loaded & need, need);
    if (L.kv_len != h->kv_len)
      return fail(h, DEC_ERR_STATE, "layer %d KV length %d differs from %d", l, L.kv_len, h->kv_len);
  }
  if (pos != h->kv_len) return fail(h, DEC_ERR_POS, "pos %d != KV length %d", pos, h->kv_len);
  if (pos >= h->d.max_ctx) return fail(h, DEC_ERR_CTX, "pos %d >= max_ctx %d", pos, h->d.max_ctx);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc;
  if (h->graph) {
    rc = h->exec ? patch_io(h, emb, out) : capture(h, emb, out);
    if (rc) return rc;
    cudaError_t e = cudaGraphLaunch(h->exec, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaGraphLaunch");
  } else {
    rc = enqueue_step(h, emb, out, s, false);
    if (rc) return rc;
  }
  h->kv_len = pos + 1;
  for (LayerDev& L : h->layers) L.kv_len = pos + 1;
  return DEC_OK;
}

int dec_set_tap(dec_handle* h, float* per_layer_out, int8_t* qact_tap, float* qscale_tap) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if ((qact_tap || qscale_tap) && h->d.weight_fmt != DEC_W_Q4B32)
    return fail(h, DEC_ERR_ARG, "int8 activation taps need DEC_W_Q4B32");
  h->tap = per_layer_out;
  h->qtap = qact_tap;
  h->qstap = qscale_tap;
  drop_graph(h);
  return DEC_OK;
}

int dec_set_dot_tap(dec_handle* h, int layer, int kernel, int32_t* dots) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (dots && (!h->fused || h->d.weight_fmt != DEC_W_Q4B32))
    return fail(h, DEC_ERR_STATE, "block-dot taps need the fused plan with int4 weights");
  if (dots && (layer < 0 || layer >= h->d.n_layers || (kernel != 0 && kernel != 2 && kernel != 3 &&
                                                        kernel != 4)))
    return fail(h, DEC_ERR_ARG, "bad layer %d / kernel %d for a block-dot tap", layer, kernel);
  h->dot_tap = dots;
  h->dot_layer = dots ? layer : -1;
  h->dot_kernel = dots ? kernel : -1;
  drop_graph(h);
  return DEC_OK;
}

int dec_set_timeline(dec_handle* h, uint64_t* buf) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (buf && !h->fused) return fail(h, DEC_ERR_STATE, "the timeline probe needs a fused plan");
  h->timeline = buf;
  drop_graph(h);
  return DEC_OK;
}

int dec_sync_status(dec_handle* h, dec_stream_t stream) {
  if (!h) {  // the no-alloc attention's flag (it has no handle)
    int flag = 0;
    const int rc = noalloc_sync_status(reinterpret_cast<cudaStream_t>(stream), &flag);
    if (rc == DEC_ERR_DEVICE)
      return fail(nullptr, rc, "dec_attention_noalloc gave up a bounded wait (flags 0x%x)", flag);
    if (rc != DEC_OK) return fail(nullptr, rc, "reading the no-alloc attention's error flag failed");
    return DEC_OK;
  }
  TLD_CUDA(h, cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  int flag = 0;
  TLD_CUDA(h, cudaMemcpy(&flag, h->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  if (flag) {
    int line = 0;
    TLD_CUDA(h, cudaMemcpy(&line, h->d_err + 1, sizeof(int), cudaMemcpyDeviceToHost));
    TLD_CUDA(h, cudaMemset(h->d_err, 0, 2 * sizeof(int)));
    if (flag & ERR_BOUNDS)
      return fail(h, DEC_ERR_DEVICE, "an index check failed (flags 0x%x, source line %d)", flag, line);
    return fail(h, DEC_ERR_DEVICE, "a kernel gave up a bounded wait (flags 0x%x)", flag);
  }
  return DEC_OK;
}

int dec_check_guards(dec_handle* h) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (!h->guards) return fail(h, DEC_ERR_STATE, "the handle was created without DEC_DEBUG_GUARDS");
  TLD_CUDA(h, cudaDeviceSynchronize());
  std::vector<uint8_t> buf;
  for (size_t i = 0; i < h->guard_list.size(); ++i) {
    const auto& g = h->guard_list[i];
    if (g.bytes == 0) continue;
    // the band before, and the pattern from the end of the user bytes to the
    // end of the band after
    const size_t after = ((g.bytes + 255) & ~(size_t)255) - g.bytes + kGuardBytes;
    for (int side = 0; side < 2; ++side) {
      const size_t n = side ? after : kGuardBytes;
      const uint8_t* src = side ? g.user + g.bytes : g.user - kGuardBytes;
      buf.resize(n);
      TLD_CUDA(h, cudaMemcpy(buf.data(), src, n, cudaMemcpyDeviceToHost));
      for (size_t j = 0; j < n; ++j)
        if (buf[j] != kGuardPattern)
          return fail(h, DEC_ERR_DEVICE, "guard band %s allocation %zu (%zu bytes) overwritten at byte %zd",
                      side ? "after" : "before", i, g.bytes,
                      side ? (ssize_t)j : (ssize_t)j - (ssize_t)kGuardBytes);
    }
  }
  // every cache row past the KV length still holds the poison it was created with
  const dec_model_desc& d = h->d;
  const size_t row = 2 * (size_t)d.head_dim;
  for (int l = 0; l < d.n_layers; ++l) {
    const LayerDev& L = h->layers[l];
    if (L.kv_len >= d.max_ctx) continue;
    int rc = for_kv_runs(h, L.kv_len, d.max_ctx, [&](int64_t off, int rows, int64_t src_row) -> int {
      buf.resize(row * rows);
      for (const uint16_t* c : {L.kc, L.vc}) {
        TLD_CUDA(h, cudaMemcpy(buf.data(), c + off, row * rows, cudaMemcpyDeviceToHost));
        for (size_t j = 0; j < buf.size(); ++j)
          if (buf[j] != 0xFF) {
            const int g = (int)(src_row / (d.max_ctx - L.kv_len));
            const int t = L.kv_len + (int)(src_row % (d.max_ctx - L.kv_len)) + (int)(j / row);
            return fail(h, DEC_ERR_DEVICE, "layer %d KV head %d: row %d past the KV length %d written",
                        l, g, t, L.kv_len);
          }
      }
      return DEC_OK;
    });
    if (rc) return rc;
  }
  return DEC_OK;
}

int dec_get_info(const dec_handle* h, dec_info* info) {
  if (!h || !info) return DEC_ERR_ARG;
  info->kernels_per_layer = h->persistent ? 1 : h->fused ? kernels_per_layer(h)
                            : h->d.weight_fmt == DEC_W_Q4B32 ? kUnfusedKernelsPerLayerQ4
                                                             : kUnfusedKernelsPerLayer;
  info->kernels_per_token = h->persistent ? 1 : info->kernels_per_layer * h->d.n_layers;
  info->n_sm = h->n_sm;
  info->kv_len = h->kv_len;
  info->weight_bytes = h->weight_bytes;
  info->kv_bytes = h->kv_bytes;
  info->workspace_bytes = h->ws_bytes;
  info->attn_grid = h->fused && !h->persistent ? fused_att_grid(h) : h->att_grid;
  info->attn_cluster = h->fused && !h->persistent ? h->att_cluster : 0;
  info->page_rows = h->paged ? h->page_rows : 0;
  info->n_pages = h->paged ? h->n_pages : 0;
  return DEC_OK;
}

int dec_launch_kernel(dec_handle* h, int kernel, int first_layer, int count, dec_stream_t stream) {
  if (!h) return fail(nullptr, DEC_ERR_ARG, "handle is NULL");
  if (!h->fused || h->persistent)
    return fail(h, DEC_ERR_STATE, "single-kernel launches need a fused plan of several kernels");
  if (kernel < 0 || kernel >= kernels_per_layer(h) || count < 0 || first_layer < 0 ||
      first_layer >= h->d.n_layers)
    return fail(h, DEC_ERR_ARG, "bad kernel / layer / count");
  const uint32_t need = required_mask(h->d);
  for (const LayerDev& L : h->layers)
    if ((L.loaded & need) != need) return fail(h, DEC_ERR_STATE, "weights not all loaded");
  if (h->kv_len >= h->d.max_ctx) return fail(h, DEC_ERR_CTX, "KV cache full");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int i = 0; i < count; ++i) {
    int rc = enqueue_fused_kernel(h, kernel, (first_layer + i) % h->d.n_layers, nullptr, nullptr,
                                  false, s);
    if (rc) return rc;
  }
  return DEC_OK;
}

int dec_destroy(dec_handle* h) {
  if (!h) return DEC_OK;
  cudaDeviceSynchronize();
  drop_graph(h);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  for (void* p : h->allocs)
    if (p) cudaFree(p);
  delete h;
  return DEC_OK;
}

const char* dec_last_error(const dec_handle* h) {
  return h ? h->err.c_str() : g_create_error.c_str();
}

}  // extern "C"
