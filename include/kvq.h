/*
 * kvq.h — C ABI of the low-bit KV-cache decode-attention library (libkvq.so).
 *
 * The library computes single-token decode attention over an asymmetrically
 * quantized KV cache, as defined by KIVI ("KIVI: A Tuning-Free Asymmetric 2bit
 * Quantization for KV Cache", papercache.org page, sections "方法细节" and
 * "附录细节", Algorithm 1), generalised to the mixed-precision window layout
 * of WindowQuant ("WindowQuant: Mixed-Precision KV Cache Quantization Based on
 * Window-Level Similarity for VLMs", ebiotrade.com page, §3.1 and §3.3).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensors are caller-owned device memory (the library allocates
 *   nothing).  fp16 means IEEE binary16, u8 means unsigned bytes.  Every
 *   device pointer must be 16-byte aligned.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every call that launches work is asynchronous on that stream, except
 *   kvq_window_assign and kvq_window_assign_eq8, which return host arrays and
 *   therefore synchronize it.
 * - Arguments are validated on the host before anything is launched; a
 *   rejected call returns a negative kvq_status, launches nothing and leaves
 *   the cache struct untouched.  After a launch, a CUDA launch error maps to
 *   KVQ_ERR_CUDA.  No entry point traps, aborts or throws.
 * - Lengths (nk, nv, nkr, nvr, ring starts) live in the host struct and are
 *   uniform over the batch and the kv heads.  The library updates them.
 *
 * Quantizer (KIVI "方法细节", first formula; WindowQuant §3.3.3 Eq.14 and 16)
 * ---------------------------------------------------------------------------
 * For a group of fp16 values x_1..x_n and b bits (qmax = 2^b - 1):
 *   mn = min x_i, mx = max x_i                      (exact, fp16 values)
 *   s32 = (mx - mn) / qmax                           (IEEE fp32 subtract, divide)
 *   s = fp16_round_nearest_even(s32), z = mn         (both stored as fp16)
 *   code_i = 0 if s == 0, else clamp(rint((x_i - z) / s), 0, qmax)
 *            (fp32 subtract and IEEE divide, rint = round half to even)
 *   dequantized value = code * s + z
 * With zero_point = KVQ_ZERO_INT (WindowQuant §3.3.3 Eq.14-16, integer zero
 * point, qmin = 0), for s != 0:
 *   zi = -rint(mn / s)                              (IEEE fp32 divide)
 *   code_i = clamp(rint(x_i / s) + zi, 0, qmax)     (IEEE fp32 divide)
 *   stored zero z = fp16_round_nearest_even(-(s * zi))   (fp32 product)
 * so that the dequantized value s (code - zi) is read as code * s + z, the
 * same form as above (z carries fp16 rounding of s * zi); for s == 0 the codes
 * are 0 and z = mn, as above.
 * K is quantized per channel over groups of `group` consecutive tokens; V is
 * quantized per token over groups of `group_v` consecutive channels (group_v
 * = 0 means group_v = group).
 *
 * Packed code layout (identical for K and V)
 * ------------------------------------------
 * Token-major rows of d_h*bits/8 bytes.  The code of channel c sits at bit
 * offset c*bits of the row read as a little-endian bit string, i.e. in byte
 * (c*bits)/8 at bit (c*bits)%8, least significant bit first.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  /* The K residual holds resid_cap tokens: call kvq_flush_residual
   * (KIVI Algorithm 1, decoding branch "len(X_Kr) == R"). */
  KVQ_FLUSH_DUE = 1,
  KVQ_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size, bad state */
  KVQ_ERR_UNSUPPORTED = -2, /* valid but not built: e.g. d_h not 64/128 */
  KVQ_ERR_CAPACITY = -3,    /* a segment or the residual ring would overflow */
  KVQ_ERR_CUDA = -4,        /* a CUDA call failed; see kvq_last_error_string */
  KVQ_ERR_WORKSPACE = -5    /* workspace missing or smaller than required */
} kvq_status;

/* Residual policies. */
enum {
  /* KIVI Algorithm 1: K tokens wait in the fp16 ring until it holds
   * resid_cap tokens, then the whole block is quantized per channel; V keeps
   * the newest resid_cap tokens in fp16 and quantizes each evicted token. */
  KVQ_POLICY_KIVI = 0,
  /* WindowQuant §3.1: text and generated tokens stay fp16; the ring is never
   * flushed and an append past resid_cap fails with KVQ_ERR_CAPACITY. */
  KVQ_POLICY_FP16_TAIL = 1
};

/* Zero points of the quantizer (see "Quantizer" above). */
enum {
  KVQ_ZERO_MIN = 0, /* KIVI: z = min of the group, a float */
  KVQ_ZERO_INT = 1  /* WindowQuant Eq.16: integer zero point */
};

#define KVQ_MAX_SEGMENTS 8

/* One packed segment: a run of tokens quantized at one bit width.  KIVI uses
 * one segment; WindowQuant uses one per width, windows of equal width made
 * contiguous (WindowQuant §3.3.1).  All buffers device, caller-owned. */
typedef struct kvq_segment {
  int32_t bits;     /* 2, 4 or 8 */
  int32_t capacity; /* tokens the buffers hold; a multiple of group */
  int32_t nk;       /* valid packed K tokens (multiple of group) */
  int32_t nv;       /* valid packed V tokens */
  void* k_codes;    /* u8   [batch][h_kv][capacity][d_h*bits/8] */
  void* k_scale;    /* fp16 [batch][h_kv][capacity/group][d_h] */
  void* k_zero;     /* fp16 [batch][h_kv][capacity/group][d_h] */
  void* v_codes;    /* u8   [batch][h_kv][capacity][d_h*bits/8] */
  void* v_scale;    /* fp16 [batch][h_kv][capacity][d_h/group_v] */
  void* v_zero;     /* fp16 [batch][h_kv][capacity][d_h/group_v] */
} kvq_segment;

/* The cache: packed segments plus one fp16 residual ring for K and one for V.
 * Residual token i (0 <= i < nkr) of K sits in ring slot
 * (k_ring_start + i) % resid_cap; likewise for V.  The token sequence that
 * attention sees is seg[0] packed, seg[1] packed, ..., then the ring, for K
 * and for V alike; K and V must describe the same number of tokens, and every
 * segment but the last must have nk == nv. */
typedef struct kvq_cache {
  int32_t batch;     /* b */
  int32_t h_kv;      /* kv heads */
  int32_t h_q;       /* query heads; a multiple of h_kv (GQA when larger) */
  int32_t d_h;       /* head dim: 64 or 128 */
  int32_t group;     /* G: K quantization group in tokens (also V's, see group_v) */
  int32_t resid_cap; /* R: ring capacity in tokens, a multiple of group */
  int32_t policy;    /* KVQ_POLICY_* */
  float sm_scale;    /* softmax scale applied to q.k (1/sqrt(d_h) typical) */
  int32_t n_seg;     /* 1..KVQ_MAX_SEGMENTS */
  kvq_segment seg[KVQ_MAX_SEGMENTS];
  void* k_resid;     /* fp16 [batch][h_kv][resid_cap][d_h] */
  void* v_resid;     /* fp16 [batch][h_kv][resid_cap][d_h] */
  int32_t nkr, nvr;  /* residual K / V tokens */
  int32_t k_ring_start, v_ring_start; /* ring slot of the oldest residual token */
  int32_t zero_point; /* KVQ_ZERO_MIN (0, the default) or KVQ_ZERO_INT */
  int32_t group_v;    /* V quantization group in channels, a power of two
                         dividing d_h, at least 8; 0 = group (WindowQuant
                         §3.3.3: K groups of one window, S tokens, beside
                         per-token V groups) */
} kvq_cache;

/* WindowQuant ingest plan (WindowQuant §3.1 Eq.7 windows, §3.3.1 reorder).
 * The T input tokens are n_windows windows of `window` tokens followed by a
 * tail of T - n_windows*window tokens.  Windows are written in the order
 * perm[0], perm[1], ...; a window of width 2/4/8 is appended to the first
 * segment with that width (K quantized per channel over groups of `group`
 * tokens inside the window, V per token); a width-16 window and the tail go
 * to the fp16 ring.  Host arrays, read during the call only. */
typedef struct kvq_window_plan {
  int32_t window;      /* S, a multiple of group */
  int32_t n_windows;
  const int8_t* bits;  /* [n_windows], each 2, 4, 8 or 16 */
  const int32_t* perm; /* [n_windows], a permutation of 0..n_windows-1 */
} kvq_window_plan;

/* Append T new tokens of K and V (fp16 [batch][h_kv][T][d_h], device).
 *
 * plan == NULL, policy KIVI: the T tokens go through KIVI Algorithm 1 one by
 *   one (prefill when the cache is empty is the same as T decode appends):
 *   - V: pushed into the ring; whenever it would exceed resid_cap, the oldest
 *     token is quantized per token and appended to the last segment
 *     ("值缓存的队列式更新机制");
 *   - K: pushed into the ring; every time the ring reaches resid_cap, the
 *     block is quantized per channel and appended to the last segment
 *     ("键缓存的流式更新与注意力计算") -- except when the ring is full after
 *     the last token: then the block is left in place and the call returns
 *     KVQ_FLUSH_DUE, so the caller chooses when to run kvq_flush_residual.
 * plan == NULL, policy FP16_TAIL: the tokens go to the ring only.
 * plan != NULL: WindowQuant ingest as described at kvq_window_plan.
 *
 * Returns KVQ_OK or KVQ_FLUSH_DUE on success; KVQ_ERR_CAPACITY if a segment or
 * the ring would overflow (nothing is launched).  The cache struct's lengths
 * are updated on success. */
kvq_status kvq_quantize_append(kvq_cache* cache, const void* k_new,
                               const void* v_new, int32_t T,
                               const kvq_window_plan* plan, void* stream);

/* Quantize the oldest floor(nkr/group)*group residual K tokens per channel
 * (groups of `group` tokens) and append them to the last segment's packed K
 * (KIVI Algorithm 1: "if len(X_Kr) == R: ... KeyQuant ... X_Kr = empty").
 * Returns KVQ_OK (also when nothing is due). */
kvq_status kvq_flush_residual(kvq_cache* cache, void* stream);

/* Bytes of device workspace kvq_decode_attention needs when it may split each
 * (batch, kv head) over at most max_splits CTAs (1..KVQ_MAX_SPLITS). */
#define KVQ_MAX_SPLITS 128
size_t kvq_workspace_bytes(const kvq_cache* cache, int32_t max_splits);

/* Zero-fill a workspace before its first use (cudaMemsetAsync).  Every later
 * call of kvq_decode_attention leaves it ready for the next. */
kvq_status kvq_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* Decode attention for one new query token per head (KIVI Algorithm 1,
 * decoding branch; WindowQuant §3.3.1 for several segments):
 *   a_t = sm_scale * q . k_t over every cached token t (dequantized packed K
 *         or fp16 residual K), p = softmax(a), out = sum_t p_t v_t
 *         (dequantized packed V or fp16 residual V).
 * q fp16 [batch][h_q][d_h], out fp16 [batch][h_q][d_h] (device).  Query head
 * j reads kv head j / (h_q / h_kv).  The work is split over the token axis
 * (split-K, FlashDecoding style) and merged by the last CTA of each head.
 * workspace: device, at least kvq_workspace_bytes(cache, 1) bytes, zeroed
 * once by kvq_workspace_init; more workspace allows more splits.  Calls that
 * share a workspace must not overlap on the GPU.  With zero tokens cached the
 * output is zero. */
kvq_status kvq_decode_attention(const kvq_cache* cache, const void* q,
                                void* out, void* workspace, size_t ws_bytes,
                                void* stream);

/* Order of a decode step's attention and its due K flush. */
typedef enum {
  KVQ_STEP_ATTEND_FIRST = 0, /* attention over the ring of R fp16 K tokens, then the flush */
  KVQ_STEP_FLUSH_FIRST = 1   /* the flush, then the attention (KIVI Algorithm 1's order) */
} kvq_step_order;

/* One decode step of KIVI Algorithm 1's decoding branch (KIVI page,
 * "附录细节" Algorithm 1): the new token of every (batch, kv head) is appended
 * as by kvq_quantize_append with T = 1 (k_new, v_new fp16
 * [batch][h_kv][1][d_h]); the K flush that the append made due runs as by
 * kvq_flush_residual, and decode attention as by kvq_decode_attention (q,
 * out, workspace: as there).  `order` KVQ_STEP_FLUSH_FIRST is Algorithm 1's
 * order (a K ring that reached R is quantized before the attention);
 * KVQ_STEP_ATTEND_FIRST attends over the state the append left (R fp16 K
 * tokens) and flushes after.  The results equal those of the three calls
 * in the same order.  The kernels are chained with programmatic dependent
 * launch: each starts while the previous one ends; the attention's chunks
 * that hold no token the append or the flush writes start at once; the
 * flush takes the step's new token from k_new (unchanged until the step
 * completes), and after the attention it runs beside the attention's last
 * warps.  Asynchronous on `stream`.  Returns KVQ_OK, or a negative status
 * (KVQ_ERR_INVALID_ARG also for an unknown order); if a launch fails after
 * the append was enqueued the cache's host lengths are restored, but the
 * device writes already enqueued (ring slot, evicted V row, flushed rows)
 * happen. */
kvq_status kvq_decode_step(kvq_cache* cache, const void* k_new, const void* v_new, const void* q,
                           void* out, void* workspace, size_t ws_bytes, int32_t order, void* stream);

/* kvq_decode_step fed from host memory: the step's inputs are copied from
 * host_in to dev_in, the step runs on them, and its output is copied from
 * dev_out to host_out, all enqueued on `stream` (asynchronous: synchronize
 * the stream before reading host_out).
 *   host_in, dev_in  fp16 [new K: batch*h_kv*d_h | new V: batch*h_kv*d_h |
 *                    q: batch*h_q*d_h], contiguous (the K and V parts in the
 *                    [batch][h_kv][1][d_h] layout of kvq_decode_step)
 *   host_out         fp16 [batch][h_q][d_h]; dev_out device, the same shape
 * Host buffers should be page-locked for the copies to be asynchronous;
 * device buffers 16-byte aligned.  workspace, ws_bytes, order: as for
 * kvq_decode_step.  Returns what kvq_decode_step returns, or
 * KVQ_ERR_INVALID_ARG / KVQ_ERR_CUDA for the arguments and the copies. */
kvq_status kvq_decode_step_host(kvq_cache* cache, const void* host_in, void* host_out, void* dev_in,
                                void* dev_out, void* workspace, size_t ws_bytes, int32_t order,
                                void* stream);

/* Device error word of a workspace (0 = none; nonzero = a bounded wait timed
 * out inside a kernel).  Synchronizes `stream`. */
kvq_status kvq_workspace_error(const void* workspace, int32_t* err_out,
                               void* stream);

/* WindowQuant window bit-width assignment and reorder (WindowQuant §3.2.1
 * Eq.7-8 similarity, §3.3.1 reorder), with the rank rule of this library:
 *   keys      fp16 [batch][h_kv][M][d_h] (vision-token keys, device)
 *   text_keys fp16 [batch][h_kv][N][d_h] (text-token keys, device)
 * Window w holds vision tokens [w*S, w*S+S) for w < n_windows = M / S.  Its
 * score is the mean over the batch of cos(sum of its keys, sum of the text
 * keys), each sum taken over tokens of the concatenated h_kv*d_h key vector.
 * Windows are ranked by score (ties: lower index first); the first
 * floor(frac8*n) get 8 bits, the next floor(frac4*n) 4 bits, the rest 2 bits,
 * where n counts the ranked windows.  first_window_fp16 != 0 gives window 0
 * width 16 and leaves it out of the ranking (WindowQuant §3.2.2).
 * perm_out lists windows by width descending, index ascending within a
 * width (the ingest order of kvq_window_plan).
 * bits_out int8 [n_windows], perm_out int32 [n_windows], sim_out double
 * [n_windows] or NULL: host memory.  workspace: device, at least
 * kvq_window_assign_workspace_bytes(...) bytes, no initialization needed. */
size_t kvq_window_assign_workspace_bytes(int32_t batch, int32_t h_kv,
                                         int32_t d_h, int32_t M, int32_t S);
kvq_status kvq_window_assign(const void* keys, const void* text_keys,
                             int32_t batch, int32_t h_kv, int32_t d_h,
                             int32_t M, int32_t S, int32_t N, float frac8,
                             float frac4, int32_t first_window_fp16,
                             void* workspace, size_t ws_bytes, int8_t* bits_out,
                             int32_t* perm_out, double* sim_out, void* stream);

/* WindowQuant window bit widths as the page defines them (WindowQuant §3.2.1
 * Eq.8, §3.2.2, §3.2.3 Eq.10-11), and the reorder of §3.3.1:
 *   vision fp16 [batch][M][dim] (vision-token embeddings, device)
 *   text   fp16 [batch][N][dim] (text-token embeddings, device)
 * Window w holds vision tokens [w*S, w*S+S) for w < n_windows = M / S (a tail
 * M mod S stays FP16 at ingest).  Per request b and window w, Eq.8:
 *   sim = 1/(S N) sum_j sum_k t_j . w_k / (|t_j| |w_k|)   (a zero token adds 0)
 * as (sum_j t_j / |t_j|) . (sum_k w_k / |w_k|) / (S N): products in fp32 (exact
 * for fp16 squares), sums of at most 16 terms in fp32 inside fp64 sums, so a
 * score carries a relative error of about 1e-7 (a window within that of a
 * threshold can fall either side).  dim must be a multiple of 8.  Thresholds from the layer similarity s (Eq.9, given by
 * the caller) and alpha (nonzero): T_low = (e^(alpha s) - 1) / (e^alpha - 1),
 * T_high = (e^(-alpha s) - 1) / (e^(-alpha) - 1).  A request puts window w at
 * 16 bits if sim > T_high, 2 bits if sim < T_low, else 4 bits; the batch takes
 * the most frequent choice, a tie going to the wider width; first_window_fp16
 * != 0 pins window 0 to 16 bits.  perm_out lists windows by width descending,
 * index ascending (the ingest order of kvq_window_plan; 16-bit windows go to
 * the fp16 ring).  bits_out int8 [n_windows], perm_out int32 [n_windows],
 * sim_out double [batch][n_windows] or NULL: host memory.  workspace: device,
 * at least kvq_window_assign_eq8_workspace_bytes(...) bytes, no
 * initialization needed.  Synchronizes `stream`. */
size_t kvq_window_assign_eq8_workspace_bytes(int32_t batch, int32_t dim,
                                             int32_t M, int32_t S, int32_t N);
kvq_status kvq_window_assign_eq8(const void* vision, const void* text,
                                 int32_t batch, int32_t dim, int32_t M,
                                 int32_t S, int32_t N, double layer_sim,
                                 double alpha, int32_t first_window_fp16,
                                 void* workspace, size_t ws_bytes,
                                 int8_t* bits_out, int32_t* perm_out,
                                 double* sim_out, void* stream);

/* Paged cache with per-sequence lengths (no counterpart in the pages: the
 * KIVI page names a combination with PagedAttention-style memory management
 * as future work, "局限性与未来工作").
 *
 * Each sequence of the batch runs KIVI Algorithm 1 on its own: its lengths
 * (packed K/V tokens, ring tokens, ring starts) are kept per sequence in the
 * host struct, so sequences of different lengths share one launch.  Packed
 * tokens live in a pool of pages of `page_tokens` tokens; page j of
 * sequence b holds its packed tokens [j*P, j*P+P) (P = page_tokens) and is
 * the pool page block_table[b*max_pages + j].  One pool page holds every kv
 * head:
 *   k_codes u8   [n_pages][h_kv][P][d_h*bits/8]
 *   k_scale fp16 [n_pages][h_kv][P/group][d_h]     (k_zero alike)
 *   v_codes u8   [n_pages][h_kv][P][d_h*bits/8]
 *   v_scale fp16 [n_pages][h_kv][P][d_h/group_v]   (v_zero alike)
 * The codec, the packed row format and the policy are those of kvq_cache
 * with one segment and policy KVQ_POLICY_KIVI.  The fp16 rings are per
 * sequence: k_resid/v_resid fp16 [batch][h_kv][resid_cap][d_h].
 *
 * The block table is device memory, owned and filled by the caller, who
 * maps a sequence's pages before its packed tokens reach them (the host
 * checks that the mapped extent, max_pages*P tokens, is not exceeded).
 * The kernels read the table and check every entry: an entry outside
 * 0..n_pages-1 is not followed (pool page 0 is read instead and nothing
 * is written), and the device word `err` is set to 2; read it with
 * kvq_workspace_error(err, ...).  A sequence with no tokens gets a zero
 * output. */
#define KVQ_MAX_SEQS 256

typedef struct kvq_seq_state {
  int32_t nk, nv;                      /* packed K / V tokens */
  int32_t nkr, nvr;                    /* fp16 ring K / V tokens */
  int32_t k_ring_start, v_ring_start;  /* ring slot of the oldest ring token */
} kvq_seq_state;

typedef struct kvq_paged_cache {
  int32_t batch;       /* sequences, 1..KVQ_MAX_SEQS */
  int32_t h_kv, h_q, d_h;
  int32_t group;       /* G (K groups, tokens), a power of two 16..256 */
  int32_t group_v;     /* V groups (channels); 0 = group */
  int32_t resid_cap;   /* R, a multiple of group */
  int32_t bits;        /* 2, 4 or 8 */
  int32_t zero_point;  /* KVQ_ZERO_MIN or KVQ_ZERO_INT */
  int32_t page_tokens; /* P, a multiple of 128 and of group */
  int32_t n_pages;     /* pages in the pool */
  int32_t max_pages;   /* columns of the block table */
  float sm_scale;
  void *k_codes, *k_scale, *k_zero, *v_codes, *v_scale, *v_zero; /* pool */
  const int32_t* block_table; /* device int32 [batch][max_pages] */
  void* k_resid;       /* fp16 [batch][h_kv][resid_cap][d_h] */
  void* v_resid;
  int32_t* err;        /* device int32 error word, zeroed by the caller */
  kvq_seq_state seq[KVQ_MAX_SEQS];
} kvq_paged_cache;

/* Append new tokens per sequence (KIVI Algorithm 1, as kvq_quantize_append
 * with plan == NULL and policy KIVI, each sequence on its own): k_new, v_new
 * fp16 [batch][h_kv][T][d_h] (device); sequence b takes its first t_seq[b]
 * rows (host int32 [batch], each 0..T; NULL = T for every sequence).
 * Returns KVQ_FLUSH_DUE when some sequence's K ring is full after its last
 * token (call kvq_paged_flush_residual), KVQ_ERR_CAPACITY (nothing launched)
 * when some sequence would pass max_pages*P packed tokens. */
kvq_status kvq_paged_append(kvq_paged_cache* cache, const void* k_new,
                            const void* v_new, int32_t T,
                            const int32_t* t_seq, void* stream);

/* For every sequence whose K ring holds resid_cap tokens (the sequences
 * that made kvq_paged_append return KVQ_FLUSH_DUE), quantize the block per
 * channel into its pages (KIVI Algorithm 1: "len(X_Kr) == R"); the other
 * sequences are left as they are. */
kvq_status kvq_paged_flush_residual(kvq_paged_cache* cache, void* stream);

/* Workspace of kvq_paged_decode_attention with at most max_splits CTAs per
 * (sequence, kv head); zero it once with kvq_workspace_init. */
size_t kvq_paged_workspace_bytes(const kvq_paged_cache* cache,
                                 int32_t max_splits);

/* Decode attention (as kvq_decode_attention) over each sequence's own
 * tokens: q, out fp16 [batch][h_q][d_h] (device).  The host splits each
 * sequence over a number of CTAs that grows with its length. */
kvq_status kvq_paged_decode_attention(const kvq_paged_cache* cache,
                                      const void* q, void* out,
                                      void* workspace, size_t ws_bytes,
                                      void* stream);

/* Decode attention without a caller workspace (no counterpart in the pages).
 *
 * Same computation, arguments and result as kvq_decode_attention, for callers
 * that cannot allocate device memory: for instance a custom-operator or
 * plugin interface that passes only the input and output tensors, or a
 * process whose device memory belongs to another allocator, where calling
 * cudaMalloc is not allowed or would stall the device.  The workspace lives
 * instead in a static array of KVQ_NOALLOC_SCRATCH_BYTES inside the library,
 * allocated once per GPU that loads the library and kept until the process
 * exits; the call allocates nothing.
 *
 * - The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 * - A cache whose batch * h_kv needs more than the array holds is rejected
 *   with KVQ_ERR_CAPACITY (kvq_last_error_string says so) before any launch.
 * - All calls share the one array, and it keeps the previous call's contents
 *   (each call clears the part that must start at zero, on `stream`).  Calls
 *   whose work can overlap on the GPU race on it: serialize them. */
#define KVQ_NOALLOC_SCRATCH_BYTES (4u << 20)
kvq_status kvq_decode_attention_noalloc(const kvq_cache* cache, const void* q,
                                        void* out, void* stream);

/* Error word of that static scratch on the current device (0 = none;
 * nonzero = a bounded wait timed out inside a decode kernel, the output is
 * not valid), as kvq_workspace_error reports it for a caller workspace.
 * Each kvq_decode_attention_noalloc call clears the word first, so read it
 * after every call whose result matters.  Synchronizes `stream`.  No
 * counterpart in the pages. */
kvq_status kvq_noalloc_error(int32_t* err_out, void* stream);

/* Static description of a status code. */
const char* kvq_status_string(kvq_status status);

/* Message of the last KVQ_ERR_CUDA / validation failure on this thread. */
const char* kvq_last_error_string(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
