/*
 * dec.h — C ABI of the batch-1 decode library (libtld_gb300.so).
 *
 * One decode step runs one token through a stack of Llama-style decoder layers
 * with a KV cache that grows by one row per step.  The per-layer op chain is
 * the one listed on "RDNA4 Decode Kernel Fusion: Pipeline Barriers, Not
 * Launches, Are the Win", section "Decode is where the bubble has nowhere to
 * go": input RMSNorm and weight multiply, QKV projection, RoPE on q and k,
 * attention against the KV cache, output projection, post-attention RMSNorm
 * and multiply, gate and up projections, SwiGLU, down projection.  The fused
 * plan runs it as five kernels per layer (the fusions of that page's FAQ and
 * of section "Fusion removes the barrier by removing the write"); the unfused
 * plan keeps one kernel per op as the ablation ("Backend-Specific Kernel
 * Fusion", section "A practical engineering example": keep the old route).
 * Per step only the position advances; a CUDA graph of the whole token is
 * captured once and replayed ("Vulkan Command Buffer Reuse vs CUDA Graphs:
 * RDNA4 Decode Overhead", section "Why NVIDIA got a free 14 percent").
 *
 * Conventions for every call:
 *   - returns DEC_OK (0) or a negative DEC_ERR_* code; the message of the last
 *     failure is kept in the handle (dec_last_error);
 *   - arguments are validated on the host, synchronously, before any work is
 *     queued; no call aborts or exits the process;
 *   - pointers marked "host or device" may point to either (CUDA unified
 *     addressing decides); pointers marked "device" must be device memory;
 *   - all calls on one handle must come from one host thread at a time.
 */
#ifndef TLD_GB300_DEC_H
#define TLD_GB300_DEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dec_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum dec_status {
  DEC_OK = 0,
  DEC_ERR_ARG = -1,    /* null pointer, bad enum, wrong byte count */
  DEC_ERR_SHAPE = -2,  /* model shape this library does not support */
  DEC_ERR_STATE = -3,  /* step before every weight / KV row is loaded */
  DEC_ERR_POS = -4,    /* pos differs from the current KV length */
  DEC_ERR_CTX = -5,    /* pos or KV length reaches max_ctx */
  DEC_ERR_CUDA = -6,   /* a CUDA runtime call failed (message kept) */
  DEC_ERR_OOM = -7,    /* device allocation failed */
  DEC_ERR_DEVICE = -8  /* a kernel gave up a bounded wait and raised its error flag */
};

enum dec_weight_fmt {
  DEC_W_BF16 = 0,  /* bf16 matrices [out][in], row-major (K contiguous) */
  DEC_W_Q4B32 = 1  /* int4 in blocks of 32 along K + one fp16 scale per block;
                      the GEMV inputs are quantized to int8 per 32-block */
};

enum dec_flags {
  DEC_PLAN_FUSED = 0,    /* five kernels per layer (default): norm + QKV + RoPE + KV append;
                            attention; o-proj + residual; norm + gate/up + SwiGLU;
                            down + residual */
  DEC_PLAN_UNFUSED = 1,  /* one kernel per op: the ablation / reference chain */
  DEC_NO_GRAPH = 2,      /* launch eagerly instead of replaying a CUDA graph */
  DEC_NO_PDL = 4,        /* fused plan: launch without programmatic dependent launch,
                            so each kernel starts only after the previous one ends */
  DEC_PLAN_PERSISTENT = 8, /* the fused layer's five phases for every layer in one
                              persistent kernel per step (one CTA per SM, grid barriers
                              between phases, one weight stream through the step) */
  DEC_NO_L2_AHEAD = 16,    /* fused plan: do not prefetch the next kernel's bytes into L2
                              at the end of each kernel's stream */
  DEC_ATTN_GLOBAL_MERGE = 32, /* five-kernel plan: attention over a flat grid whose split heads
                                 are merged through global memory by the last CTA of each head,
                                 instead of one thread-block cluster per KV head merging in
                                 distributed shared memory */
  DEC_PLAN_THREE = 64,        /* fused plan with three kernels per layer: norm + QKV + RoPE +
                                 KV append; attention + o-proj + residual; norm + gate/up +
                                 SwiGLU + down + residual (each of the last two one launch of
                                 two phases separated by a grid barrier) */
  DEC_DEBUG_GUARDS = 128,     /* memory-safety checks that need no sanitizer: every device
                                 buffer between guard bands of a known pattern, its bytes
                                 poisoned with 0xFF (NaN as fp32 and bf16) until written, KV
                                 rows past the KV length kept poisoned; dec_check_guards
                                 verifies them */
  DEC_ROPE_INTERLEAVED = 256, /* RoPE rotates dims (2i, 2i+1) of a head as pair i instead of
                                 (i, i + head_dim/2); same angles pos * theta^(-2i/head_dim) */
  DEC_PAGED_KV = 512,         /* fused plans: each layer's KV cache is a pool of pages, a page
                                 holding page_rows positions of one KV head (one attention
                                 chunk: 64 at head_dim 128, 128 at 64), laid out
                                 [page][n_kv_heads][page_rows][head_dim]; a page table maps
                                 position chunk c to page pages[c] (dec_set_page_table) */
  DEC_PLAN_FOUR = 1024,       /* fused plan with four kernels per layer: norm + QKV + RoPE + KV
                                 append; attention; o-proj + residual; norm + gate/up + SwiGLU +
                                 down + residual (one launch of two phases, grid barrier) */
  DEC_Q4_PUBLISH = 2048,      /* DEC_W_Q4B32, five- and four-kernel plans: the kernel that
                                 produces each GEMV input publishes its int8 codes once (per
                                 32-block: codes, scale, sum; RMSNorm inputs also per-CTA sums
                                 of squares), instead of every CTA of the GEMV quantizing the
                                 whole vector itself (the default) */
  DEC_FUSE_ATTN_OPROJ = 4096  /* fused plans with the cluster attention: attention and the
                                 o-projection + residual in one cluster launch; each KV head's
                                 cluster multiplies its merged output by its own columns of Wo
                                 (stored per KV-head group) and the last cluster to finish a
                                 row range adds the groups' partial vectors in group order.
                                 Four kernels per layer (three with DEC_PLAN_FOUR) */
};

/* Tensor ids for dec_load_weights.  bf16 models load the norm vectors (bf16
 * [hidden]) and the seven matrices (bf16 [out][in]).  Q4 models load the norm
 * vectors, the seven matrices as packed nibbles ([out][in/32] blocks of 16
 * bytes: element 2i in the low nibble and 2i+1 in the high nibble of byte i of
 * the block, each stored as q + 8 in [0, 15]) and, under id + DEC_T_SCALES,
 * their fp16 scales ([out][in/32]). */
enum dec_tensor {
  DEC_T_ATTN_NORM = 0, /* [hidden] */
  DEC_T_WQ = 1,        /* [n_q_heads*head_dim][hidden] */
  DEC_T_WK = 2,        /* [n_kv_heads*head_dim][hidden] */
  DEC_T_WV = 3,        /* [n_kv_heads*head_dim][hidden] */
  DEC_T_WO = 4,        /* [hidden][n_q_heads*head_dim] */
  DEC_T_FFN_NORM = 5,  /* [hidden] */
  DEC_T_WGATE = 6,     /* [ffn][hidden] */
  DEC_T_WUP = 7,       /* [ffn][hidden] */
  DEC_T_WDOWN = 8,     /* [hidden][ffn] */
  DEC_T_SCALES = 16    /* add to WQ..WDOWN for the Q4 scales */
};

typedef struct dec_model_desc {
  int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn;
  float rms_eps;      /* RMSNorm epsilon, inside the square root */
  float rope_theta;   /* RoPE base: angle of pair i at position p = p * theta^(-2i/head_dim) */
  int32_t max_ctx;    /* KV cache capacity in positions */
  int32_t weight_fmt; /* enum dec_weight_fmt */
  int32_t flags;      /* enum dec_flags, OR-ed */
} dec_model_desc;

typedef struct dec_info {
  int32_t kernels_per_layer;  /* launches per layer of the chosen plan (1 for the
                                 persistent plan, whose one launch covers every layer) */
  int32_t kernels_per_token;  /* launches per dec_step */
  int32_t n_sm;               /* SMs the grids are sized for */
  int32_t kv_len;             /* current KV length (next pos) */
  int64_t weight_bytes;       /* device bytes of all layers' weights as stored */
  int64_t kv_bytes;           /* device bytes of the KV cache (both K and V) */
  int64_t workspace_bytes;    /* device bytes of activations + split-K workspace */
  int32_t attn_grid;          /* CTAs of the attention launch (fused plan) */
  int32_t attn_cluster;       /* CTAs per KV head in one thread-block cluster, or 0 for
                                 the flat grid merged through global memory */
  int32_t page_rows;          /* DEC_PAGED_KV: positions per page (else 0) */
  int32_t n_pages;            /* DEC_PAGED_KV: pages per layer = entries of the page table */
} dec_info;

typedef struct dec_handle dec_handle; /* opaque */

/* Source: "Vulkan Command Buffer Reuse vs CUDA Graphs: RDNA4 Decode Overhead",
 * section "Why NVIDIA got a free 14 percent" (build the launch structure once,
 * reuse it every token); the shapes are those of a Llama-style decoder layer
 * ("RDNA4 Decode Kernel Fusion", section "Decode is where the bubble has
 * nowhere to go").
 * Validates the shape and allocates every device buffer (weights, KV cache,
 * workspaces) on the current CUDA device.  Supported: head_dim 64 or 128,
 * n_q_heads a multiple of n_kv_heads, hidden and ffn multiples of 8 (of 32
 * for DEC_W_Q4B32), 1 <= max_ctx <= 65536.  *out is NULL on failure. */
int dec_create(const dec_model_desc* desc, dec_handle** out);

/* Source: the layer's weights as the op chain names them ("RDNA4 Decode Kernel
 * Fusion", section "Decode is where the bubble has nowhere to go"), in bf16 or
 * in int4 blocks of 32 with an fp16 scale (the block-quantized workload this
 * library is measured on).
 * Copies one tensor of one layer (host or device src, `bytes` long, layout as
 * in enum dec_tensor) into library-owned device memory, repacking it into the
 * kernels' tiled layout.  Blocks until done.  The caller keeps src. */
int dec_load_weights(dec_handle* h, int layer, int tensor, const void* src, size_t bytes);

/* Source: none on the pages; an addition the measured workloads force (every
 * one starts from a KV cache prefilled to 127, 1023, 2047 or 4095 positions).
 * Loads the first n_pos cache rows of one layer: k and v are host or device
 * bf16 [n_kv_heads][n_pos][head_dim] (k already rotated by RoPE at its own
 * position, v raw).  Sets that layer's KV length to n_pos.  Blocks until done
 * and waits for all queued work of the device first. */
int dec_load_kv(dec_handle* h, int layer, const void* k_bf16, const void* v_bf16, int n_pos);

/* Source: "RDNA4 Decode Kernel Fusion", section "What it does to the token",
 * Table 1 (the token ends with "LM head + sampling" after the layers).
 * Loads the LM head: final_norm_bf16, host or device bf16 [hidden], the
 * final RMSNorm weight, and w_bf16, host or device bf16 [vocab][hidden]
 * ([out][in], row-major), copied (repacked) into library-owned memory.
 * vocab must be a positive multiple of 4.  Blocks until done; discards the
 * captured graph.  Tokens are produced only once dec_set_token_out is given a
 * destination. */
int dec_load_lm_head(dec_handle* h, const void* final_norm_bf16, const void* w_bf16, int vocab);

/* Source: as dec_load_lm_head.  token_out: device int32, or NULL to stop
 * producing tokens.  While set, every dec_step ends with the LM head: the
 * final RMSNorm (the model's eps) of the step's out_hidden times the final
 * norm weight, logits = W n in fp32, and the greedy token, the index of the
 * largest logit (the lowest index among equal ones), written to *token_out.
 * logits_tap (device fp32 [vocab] or NULL) also receives the logits.  The
 * choice is the same every run: each CTA's largest logit is combined with an
 * order-independent maximum.  Needs dec_load_lm_head first (DEC_ERR_STATE);
 * discards the captured graph. */
int dec_set_token_out(dec_handle* h, int32_t* token_out, float* logits_tap);

/* Source: "Kernel fusion and block bridging", section "Fusion" (the rotated k
 * and the v of a token written into their KV pages by the projection launch).
 * Sets the page table of a DEC_PAGED_KV handle: pages, host or device int32
 * [n], n = n_pages (dec_get_info), a permutation of 0..n-1; position chunk c
 * lives in page pages[c] of every layer's pool.  Rows already in the cache
 * move with their chunks.  Waits for the device; discards nothing (the graph
 * reads the table from device memory).  DEC_ERR_STATE without DEC_PAGED_KV,
 * DEC_ERR_ARG for a wrong length, an entry out of range or repeated. */
int dec_set_page_table(dec_handle* h, const int32_t* pages, int n);

/* Source: none on the pages; an addition the parity check of the KV append
 * forces (the rows the QKV kernel wrote are compared with the reference chain's).
 * Copies rows [first_pos, first_pos + n_pos) of one layer's cache into k_bf16
 * and v_bf16, host or device bf16 [n_kv_heads][n_pos][head_dim] each (the
 * layout dec_load_kv takes).  Rows past the KV length hold whatever was last
 * written there.  Waits for all queued work of the device first; blocks until
 * done. */
int dec_read_kv(dec_handle* h, int layer, void* k_bf16, void* v_bf16, int first_pos, int n_pos);

/* Source: none on the pages; an addition for repeated measurement from the
 * same prefilled state.
 * Rewinds every layer's KV length to n_pos (<= the current length); rows past
 * it are overwritten by later steps.  Waits for the device first. */
int dec_truncate_kv(dec_handle* h, int n_pos);

/* Source: "RDNA4 Decode Kernel Fusion", section "Decode is where the bubble
 * has nowhere to go" (one token through every layer's chain) and "Vulkan
 * Command Buffer Reuse vs CUDA Graphs", section "Why NVIDIA got a free 14
 * percent" (the KV length grows by one each token; only it changes between
 * replays of the captured token).
 * One decode step, queued on `stream`, returns after enqueue.
 * token_embedding: device fp32 [hidden], the stack's input at this position.
 * out_hidden: device fp32 [hidden], the last layer's output (no final norm,
 * no LM head).  pos must equal the current KV length (strictly sequential);
 * every layer appends its k, v at row pos and attends to rows 0..pos; after
 * the call the KV length is pos + 1.  Neither buffer may be written by other
 * work until the step has run. */
int dec_step(dec_handle* h, const float* token_embedding, int pos, float* out_hidden,
             dec_stream_t stream);

/* Source: none on the pages; an addition the per-layer parity check forces
 * (the hidden state after every layer is compared with the reference chain,
 * "Backend-Specific Kernel Fusion", section "Where it breaks": define
 * tolerances and test them).
 * Debug taps (both may be NULL): per_layer_out, device fp32 [n_layers][hidden],
 * receives every layer's output at each step; qact_tap (DEC_W_Q4B32 only),
 * device int8 [n_layers][4][max(hidden, ffn, n_q_heads*head_dim)], receives
 * the int8 inputs of the q, o, gate and down projections, and qscale_tap,
 * device fp32 [n_layers][4][max(...)/32], their block scales.  Setting taps
 * discards the captured graph; it is recaptured at the next step. */
int dec_set_tap(dec_handle* h, float* per_layer_out, int8_t* qact_tap, float* qscale_tap);

/* Source: none on the pages; an addition the bit-exact check of the integer
 * block dots of the int4/int8 path forces.
 * Integer block-dot tap (fused plans, DEC_W_Q4B32): at the next steps, the
 * GEMV `kernel` (0 = QKV, 2 = o-proj, 3 = gate/up, 4 = down) in `layer`
 * writes every int32 block dot sum_{i<32} q_w * q_x into dots, device int32
 * [rows][K/32], rows in the library's tiled order (QKV: q heads then k heads
 * with dims (i, i + head_dim/2) adjacent, then v; gate/up: gate and up rows
 * alternating).  NULL turns it off.  Discards the captured graph.  For the
 * bit-exact check of the integer path against the int8 input tap. */
int dec_set_dot_tap(dec_handle* h, int layer, int kernel, int32_t* dots);

/* Source: "RDNA4 Decode Kernel Fusion", section "What I am building next"
 * (measure with GPU timestamps rather than trusting the model).
 * GPU timeline probe of the fused plans (NULL turns it off): buf is device
 * uint64 [n_layers * 5][8], one row per phase of a layer (row layer * 5 + p, p
 * = 0 QKV, 1 attention, 2 o-proj, 3 gate/up, 4 down, whichever kernel runs
 * it); at every step each row records, in %globaltimer nanoseconds as atomic
 * min / max: [0] earliest CTA start (second phase of a two-phase kernel:
 * earliest arrival at its grid barrier), [1] latest end of the phase, [2] /
 * [3] earliest / latest return from griddepcontrol.wait (second phase: from
 * the grid barrier), [4] latest arrival of a CTA's first stage, [5] / [6]
 * earliest / latest end of a CTA's streaming loop, [7] earliest end.
 * The caller initialises the min slots (0, 2, 5, 7) to UINT64_MAX and the max
 * slots (1, 3, 4, 6) to 0.  With DEC_PLAN_PERSISTENT, row i is phase i of the
 * step (layer * 5 + phase) and records [0] / [1] the earliest / latest return
 * from the grid barrier before it, [2] / [3] the earliest / latest end of its
 * work, and row 0 slot [5] the earliest CTA start.
 * Setting it discards the captured graph.  For measurement only ("RDNA4
 * Decode Kernel Fusion", section "What I am building next": GPU timestamps). */
int dec_set_timeline(dec_handle* h, uint64_t* buf);

/* Source: none on the pages; the library's bounded waits report here.
 * Waits for `stream` and reports DEC_ERR_DEVICE if any kernel raised its
 * error flag (a bounded wait ran out); the flag is cleared.  With h == NULL it
 * reports the flag of dec_attention_noalloc on the current device instead
 * (read and cleared with cudaMemcpyFromSymbol / ToSymbol, which allocate
 * nothing); its message is then read with dec_last_error(NULL). */
int dec_sync_status(dec_handle* h, dec_stream_t stream);

/* Source: "Backend-Specific Kernel Fusion", section "Where it breaks" (test
 * the boundary cases); it stands in for a memory checker where none can run.
 * Waits for the device, then checks every guard band of a handle created
 * with DEC_DEBUG_GUARDS and that every KV cache row past the KV length still
 * holds its poison.  Returns DEC_OK, DEC_ERR_DEVICE (the message names the
 * buffer and byte, or the layer, head and row), DEC_ERR_STATE (no guards) or
 * DEC_ERR_CUDA.  Index checks inside the kernels are compiled into the debug
 * build of the library (TLD_DEBUG_CHECKS): a failed check skips the access,
 * raises the error flag and is reported by dec_sync_status with its source
 * line. */
int dec_check_guards(dec_handle* h);

/* Source: "Backend-Specific Kernel Fusion", section "What you can do this
 * week" (record dispatch counts alongside latency).
 * Fills *info; never fails on a valid handle. */
int dec_get_info(const dec_handle* h, dec_info* info);

/* Source: none on the pages; an addition for timing one fused kernel against
 * its bandwidth roofline.
 * Launches `count` times the fused plan's kernel `kernel` of a layer (the
 * five-kernel plan: 0 = norm+QKV+RoPE+append, 1 = attention, 2 =
 * o-proj+residual, 3 = norm+gate/up+SwiGLU, 4 = down+residual;
 * DEC_PLAN_FOUR: 0-2 as five, 3 = norm+gate/up+SwiGLU+down+residual;
 * DEC_PLAN_THREE: 0 = norm+QKV+RoPE+append, 1 = attention+o-proj+residual,
 * 2 = norm+gate/up+SwiGLU+down+residual) for layers first_layer,
 * first_layer+1, ... (mod n_layers), back to back on `stream`, on the
 * activations the last step left.
 * For timing one kernel alone; the KV length does not change and the next
 * dec_step overwrites whatever these launches wrote. */
int dec_launch_kernel(dec_handle* h, int kernel, int first_layer, int count, dec_stream_t stream);

/* Decode attention without any allocation, for callers that cannot call
 * cudaMalloc: code whose device memory all belongs to another allocator (a
 * framework's caching pool, a pre-sized arena) or that runs under a rule of no
 * allocation after start-up, since cudaMalloc can block until the device is
 * idle and fragments memory the caller manages.  The pages describe no such
 * call; it is an addition of this library.
 *
 * Runs the same split-KV GQA attention kernel as dec_step for one token:
 * q: device fp32 [n_q_heads][head_dim], already rotated by RoPE;
 * k_cache, v_cache: device bf16 [n_kv_heads][ctx_stride][head_dim] (16-byte
 * aligned); rows 0..n-1 of every KV head are attended (1 <= n <= ctx_stride);
 * o: device fp32 [n_q_heads][head_dim], softmax(q.K^T / sqrt(head_dim)) V with
 * query head h reading KV head floor(h * n_kv_heads / n_q_heads).
 * Queued on `stream`; returns after enqueue.
 *
 * Scratch: one file-scope device array of about 1 MiB (partial records of
 * heads split over CTAs, per-head counters, the position, an error flag),
 * which every GPU that loads the library holds until the process exits.  The
 * first call on each device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress) and sets the kernels' shared-memory
 * limits; make that first call before any stream capture.  Every call shares
 * the array and clears what must start at zero, so calls whose work overlaps
 * on the GPU (other streams, other threads) race and must be serialised by
 * the caller.  Limits: head_dim 64 or 128, n_kv_heads <= 64, n_q_heads /
 * n_kv_heads in {1, 2, 4, 8}, the records of one call within the array (a
 * call that would exceed it returns DEC_ERR_SHAPE), ctx_stride <= 65536.
 * Returns DEC_ERR_ARG / DEC_ERR_SHAPE for bad arguments (nothing is queued)
 * and DEC_ERR_CUDA if a launch fails.  The first-call set-up is guarded per
 * device, so concurrent first calls from several host threads are safe.  A
 * wait inside the kernel that gives up (a fault elsewhere, never in normal
 * operation) leaves o partly unwritten and sets the array's error flag; the
 * next call clears it, so read it first with dec_sync_status(NULL, stream). */
int dec_attention_noalloc(const float* q, const void* k_cache, const void* v_cache, int n_q_heads,
                          int n_kv_heads, int head_dim, int ctx_stride, int n, float* o,
                          dec_stream_t stream);

/* Source: none on the pages (resource lifetime of the C ABI).
 * Frees every device buffer and the graph; accepts NULL and partially
 * created handles.  Waits for the device first. */
int dec_destroy(dec_handle* h);

/* Source: none on the pages (error reporting of the C ABI).
 * Message of the last failed call on h ("" if none); h may be NULL, in which
 * case the message of the last failed dec_create of this thread is returned. */
const char* dec_last_error(const dec_handle* h);

#ifdef __cplusplus
}
#endif
#endif /* TLD_GB300_DEC_H */
