/*
 * bca.h -- block-causal paged attention on one GPU (sm_103a), C ABI.
 *
 * The operation is the attention of a text-diffusion decode step:
 *
 *   "Inference for Interpretable Text-Diffusion Models", section
 *   "Background" (first bullet): a token attends bidirectionally to every
 *   token of its own diffusion block, causally to tokens of earlier blocks,
 *   and never to later blocks; completed blocks are therefore cacheable.
 *   Sections "KV Cache" (prefill -> decode -> commit) and "Paged Attention"
 *   (a page table maps logical positions to fixed-size physical pages).
 *
 *   "Inference: Fewer, smaller forwards", "Advancement 1" (block-causal
 *   multi-canvas decode), "Advancement 9" (only live rows are queries),
 *   "Advancement 10"/"Advancement 11" (keys carry their absolute position;
 *   an arena of promoted rows) and "Advancement 13" (canvas c attends the
 *   contiguous prefix of positions below the end of canvas c).
 *
 * Next to the attention: "Introspective Diffusion Language Model", "3.3
 * I-DLM Serving Stack" (short causal extends over the paged cache:
 * bca_extend, the same rule with one-token blocks), and "Inference: Fewer,
 * smaller forwards", "Advancement 16" (fused QKV-post before attention:
 * bca_qkv_post; softmax-plus-argmax confidence after the LM head:
 * bca_confidence, with "Advancement 2").
 *
 * Every position p gets a block index blk(p) = -1 if p < P0, else
 * floor((p - P0) / D); a query at position i sees the key at position j iff
 * blk(j) <= blk(i).  Scores are scale * q.k (scale defaults to 1/sqrt(d)),
 * softmax over the visible keys, fp32 accumulation, bf16 output rounded to
 * nearest even.  Query head h reads key/value head h / (Hq / Hkv).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; bf16
 *    tensors are passed as void*.  Every pointer must be 16-byte aligned
 *    (bca_confidence needs only element alignment, as its section says).
 *  - Layouts (row-major, innermost last):
 *      decode Q / out          [B, D, Hq, d]       k_blk, v_blk [B, D, Hkv, d]
 *      K and V pools           [num_pages, Hkv, page_size, d] (separate tensors)
 *      page_table (int32)      [B, max_pages_per_seq]; logical position p of
 *                              sequence b lives in page page_table[b][p / S],
 *                              slot p % S.  Entries that are never touched may
 *                              hold anything (e.g. -1).
 *  - The library never allocates, frees or synchronizes (except
 *    bca_read_device_status).  Every call is asynchronous on `stream`
 *    (a cudaStream_t; NULL = legacy default stream).  Launch arguments are
 *    captured by value, so calls may be recorded into a CUDA graph.
 *  - Host-detectable errors return a negative code before anything is
 *    launched.  Errors that depend on device data (page ids, lengths) are
 *    detected by the kernels, which then skip the offending tile or sequence
 *    and record the first such error in the status word at the start of the
 *    caller's workspace; no kernel traps.  Read it with
 *    bca_read_device_status.
 *  - Workspace: caller-owned device memory of at least
 *    bca_workspace_size(dims, op) bytes, prepared once with
 *    bca_workspace_init.  Calls on the same workspace must be ordered on
 *    one stream (they share its scratch area).
 *  - head_dim must be 64 or 128; page_size a multiple of 16 in [16, 256];
 *    Hq a multiple of Hkv with Hq / Hkv <= 128; any block size D >= 1.
 */
#ifndef BCA_H_
#define BCA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BCA_ABI_VERSION 1

/* Status codes. */
#define BCA_OK 0
#define BCA_ERR_INVALID_ARG (-1)      /* bad dims or scalar argument */
#define BCA_ERR_NULL (-2)             /* a required pointer is NULL */
#define BCA_ERR_ALIGN (-3)            /* a pointer is not 16-byte aligned */
#define BCA_ERR_WORKSPACE (-4)        /* workspace NULL or too small */
#define BCA_ERR_CAPACITY (-5)         /* the request cannot fit the page table */
#define BCA_ERR_CUDA (-6)             /* a CUDA runtime/driver call failed */
#define BCA_ERR_UNSUPPORTED (-7)      /* device is not sm_100-family (tcgen05) */
#define BCA_ERR_PAGE_SHARED (-8)      /* bca_validate_page_table: page used twice */
#define BCA_ERR_PAGE_RANGE (-9)       /* bca_validate_page_table: id outside pool */
/* Device-detected (reported through the workspace status word). */
#define BCA_ERR_DEVICE_PAGE_OOB (-16) /* a page id outside [0, num_pages) */
#define BCA_ERR_DEVICE_BAD_LENGTH (-17) /* a length/position outside its range */
#define BCA_ERR_DEVICE_TIMEOUT (-18)  /* an internal wait gave up (never expected) */

/*
 * Debug checks.  With the environment variable BCA_DEBUG=1 (read at each
 * call), every entry point that takes lengths, positions or a page table
 * copies them to the host (on the call's stream, waiting for the copy) and
 * checks them before launching anything; a request that fails is refused
 * and nothing runs:
 *   BCA_ERR_INVALID_ARG  a length or position out of range for the call (a
 *                        negative prefix, a decode prefix that is not a
 *                        whole number of blocks, cu_seqlens not starting at
 *                        0 / decreasing / not ending at total_tokens / a
 *                        sequence longer than max_seqlen, two tokens of one
 *                        QKV-post writing the same cache slot, a live row
 *                        promoted twice or out of range, live_count above
 *                        max_live);
 *   BCA_ERR_CAPACITY     a range that runs past the sequence's page list;
 *   BCA_ERR_PAGE_RANGE   a page-table entry the call uses outside
 *                        [0, num_pages);
 *   BCA_ERR_PAGE_SHARED  a page the call writes that another sequence also
 *                        uses, or one page twice among one sequence's used
 *                        entries (pages that several sequences only read,
 *                        a shared prefix, are allowed).
 * Without the variable these conditions are found on the device (a page id
 * outside the pool or a position past the page list is skipped and reported
 * through the status word; shared pages are not checked).  Not meant for a
 * timed path: the copies synchronise the stream.
 */

/* Operations, for bca_workspace_size. */
#define BCA_OP_DECODE 1
#define BCA_OP_PREFILL 2
#define BCA_OP_MULTICANVAS 3
#define BCA_OP_COMMIT 4
#define BCA_OP_DECODE_MIN 5 /* smallest decode workspace: no split-KV partials */

/* Shared dimensions of one call.  `version` must be BCA_ABI_VERSION. */
typedef struct bca_dims {
  int32_t version;
  int32_t batch;             /* B: number of sequences */
  int32_t block_size;        /* D: diffusion block (decode, prefill, commit rows)
                                or canvas length C (multicanvas) */
  int32_t num_q_heads;       /* Hq */
  int32_t num_kv_heads;      /* Hkv */
  int32_t head_dim;          /* d: 64 or 128 */
  int32_t page_size;         /* S: tokens per page, multiple of 16 */
  int32_t num_pages;         /* pages in each pool */
  int32_t max_pages_per_seq; /* columns of page_table */
  float softmax_scale;       /* 0 => 1/sqrt(head_dim) */
} bca_dims;

typedef struct CUstream_st* bca_stream_t; /* == cudaStream_t */

/* Library version (BCA_ABI_VERSION). */
int bca_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* bca_status_string(int status);

/* Bytes of workspace `op` needs for these dims, or 0 if the dims are invalid.
 * Decode: a status header, a per-sequence table, the work-item list and fp32
 * partial results for splitting long prefixes across CTAs (split-KV).  Any
 * size between BCA_OP_DECODE_MIN (no partials: long prefixes are then not
 * split) and BCA_OP_DECODE (the recommended size) works; the plan kernel
 * splits only as far as the partials fit.  Multicanvas: the header and, per
 * sequence, 8 bytes for every 128 entries of page-table capacity (the key
 * position range of each arena tile).  Prefill and commit need only the
 * header. */
size_t bca_workspace_size(const bca_dims* dims, int op);

/* Zero the workspace header (status word, counters).  Call once after
 * allocating a workspace; asynchronous on `stream`. */
int bca_workspace_init(void* workspace, size_t workspace_bytes, bca_stream_t stream);

/* Synchronize `stream`, return the first device-detected error recorded in
 * the workspace since the last read (BCA_OK if none), and clear it. */
int bca_read_device_status(void* workspace, bca_stream_t stream);

/* Copy the workspace's tile counters to host memory: counters[0] = key tiles
 * processed without a mask (fully included), counters[1] = tiles processed
 * with the elementwise mask (partially included), counters[2] = tiles
 * skipped (fully excluded, never loaded).  Counters accumulate over calls
 * until bca_workspace_init.  Synchronizes `stream`. */
int bca_read_tile_counters(void* workspace, int64_t counters[3], bca_stream_t stream);

/*
 * bca_decode -- one diffusion-block decode step for a batch.
 *
 * "Inference for Interpretable Text-Diffusion Models", "KV Cache", step 2:
 * the D queries of sequence b's active block (positions P_b .. P_b+D-1,
 * P_b = prefix_len[b]) attend every key of the completed prefix 0 .. P_b-1,
 * read through the page table from the pools, and the block's own D keys
 * (k_blk/v_blk, bidirectionally).  P_b must be a multiple of D ("KV Cache",
 * step 1: the prefix is whole blocks) and P_b + D <= max_pages_per_seq * S.
 *
 * commit = 1 also performs step 3 of the same section in the same call: the
 * block's K/V bits are copied into positions [P_b, P_b+D) of the pools
 * (exactly what bca_commit_kv with start_pos = prefix_len does).  The
 * attention never reads those slots, so the result is the same either way.
 *
 * q, out: [B, D, Hq, d] bf16.  k_blk, v_blk: [B, D, Hkv, d] bf16.
 * k_pool, v_pool: pools (written only when commit = 1).
 * page_table: int32 [B, max_pages_per_seq].  prefix_len: int32 [B].
 * A sequence with an invalid prefix length is treated as P_b = 0 and
 * reported as BCA_ERR_DEVICE_BAD_LENGTH.
 */
int bca_decode(const bca_dims* dims, const void* q, const void* k_blk, const void* v_blk,
               void* k_pool, void* v_pool, const int32_t* page_table,
               const int32_t* prefix_len, void* out, int commit, void* workspace,
               size_t workspace_bytes, bca_stream_t stream);

/*
 * bca_extend -- a short causal extend over the paged cache.
 *
 * "Introspective Diffusion Language Model", "3.3 I-DLM Serving Stack" and
 * Appendix D: introspective decoding appends 2N-1 causal query tokens per
 * step (at most 9 for the short extends served by one paged attention
 * kernel instead of ragged attention + paged attention + merge).  The
 * dims' block_size is the number of new tokens n.  Query i of sequence b
 * (position P_b + i, P_b = prefix_len[b]) attends every key of the prefix
 * 0 .. P_b-1, read through the page table, and the new keys 0 .. i
 * (k_new/v_new): the block rule with one-token blocks.  P_b may be any
 * length with P_b + n <= max_pages_per_seq * S.  Any n >= 1 works; the
 * kernels are the decode step's.
 *
 * commit = 1 also copies the n new K/V rows into positions [P_b, P_b+n) of
 * the pools in the same call (the attention never reads those slots).
 *
 * q, out: [B, n, Hq, d] bf16.  k_new, v_new: [B, n, Hkv, d] bf16.  Other
 * arguments, the workspace (BCA_OP_DECODE sizes) and the errors as for
 * bca_decode.
 */
int bca_extend(const bca_dims* dims, const void* q, const void* k_new, const void* v_new,
               void* k_pool, void* v_pool, const int32_t* page_table,
               const int32_t* prefix_len, void* out, int commit, void* workspace,
               size_t workspace_bytes, bca_stream_t stream);

/*
 * bca_qkv_post -- norms, RoPE and the cache write after the QKV projection.
 *
 * "Inference: Fewer, smaller forwards", "Advancement 16" (an optional fused
 * QKV-post: RoPE, norms, arena write) and "Advancement 10" (RoPE is baked
 * into the keys at each token's true absolute position).  The dims' batch B
 * and block_size n give B * n tokens (a block per sequence, or the live rows
 * of a multicanvas step).  For each token:
 *   q, k: every head vector x becomes x * w / sqrt(mean(x^2) + eps), w of
 *         length d shared by the heads (q_norm_w / k_norm_w; NULL: no norm),
 *         then each pair (x_i, x_{i+d/2}), i < d/2, is rotated by the angle
 *         positions[t] * rope_theta^(-2i/d) (rope_theta = 0: no rotation);
 *   v:    copied bit for bit.
 * Computed in fp32 with one rounding to bf16 (nearest even) per output.
 * If write_pos is not NULL, a token with write_pos[t] >= 0 also has its
 * finished key and value rows written to cache position write_pos[t] of its
 * sequence (page page_table[b][p / S], slot p % S) and, if kv_pos is not
 * NULL, its position stored in kv_pos[page][slot] (arena mode).  The
 * outputs feed bca_decode / bca_extend (k_blk, v_blk) or bca_multicanvas
 * (the live rows).
 *
 * qkv: bf16 [B, n, Hq + 2 Hkv, d] (query heads, then key heads, then value
 * heads).  positions, write_pos: int32 [B, n] (positions may be NULL when
 * rope_theta = 0 and kv_pos is NULL).  q_norm_w, k_norm_w: bf16 [d] or
 * NULL.  q_out: bf16 [B, n, Hq, d]; k_out, v_out: bf16 [B, n, Hkv, d].
 * eps >= 0, rope_theta >= 0.  Workspace: the header (BCA_OP_COMMIT size),
 * for the status word: a write position past the page table is reported as
 * BCA_ERR_DEVICE_BAD_LENGTH, a page id outside the pool as
 * BCA_ERR_DEVICE_PAGE_OOB, and that write is skipped.
 */
int bca_qkv_post(const bca_dims* dims, const void* qkv, const int32_t* positions,
                 const void* q_norm_w, const void* k_norm_w, float eps, float rope_theta,
                 void* q_out, void* k_out, void* v_out, const int32_t* write_pos,
                 void* k_pool, void* v_pool, const int32_t* page_table, int32_t* kv_pos,
                 void* workspace, size_t workspace_bytes, bca_stream_t stream);

/*
 * bca_confidence -- the top prediction at each position and its probability.
 *
 * "Inference: Fewer, smaller forwards", "Advancement 2: tau_conf": on every
 * forward the model gives a distribution over the vocabulary at each
 * uncommitted position (the softmax of its logits); the confidence is the
 * probability of the argmax, and a position commits when it clears tau_conf.
 * "Advancement 16" lists the softmax-plus-argmax over the vocabulary as one
 * fused pass.  For each row r, with m = max_v logits[r, v]:
 *   argmax[r] = the lowest index v with logits[r, v] = m,
 *   conf[r]   = 1 / sum_v exp(logits[r, v] - m).
 * A row whose logits are all -inf gets argmax 0, conf 0; NaN logits give
 * unspecified results.
 *
 * logits: [rows, vocab] with a row stride of ld elements (ld >= vocab), bf16
 * (dtype BCA_DTYPE_BF16) or fp32 (BCA_DTYPE_F32), device memory aligned to
 * its element size (rows whose start is 16-byte aligned are read fastest).
 * argmax: int32 [rows]; conf: fp32 [rows]; device memory,
 * written once per row.  1 <= vocab < 2^31.  Needs no workspace; asynchronous
 * on `stream`; rows = 0 is a no-op.  Errors: BCA_ERR_INVALID_ARG (sizes,
 * dtype), BCA_ERR_NULL, BCA_ERR_ALIGN, BCA_ERR_UNSUPPORTED, BCA_ERR_CUDA.
 */
#define BCA_DTYPE_BF16 0
#define BCA_DTYPE_F32 1
int bca_confidence(int64_t rows, int64_t vocab, int64_t ld, int dtype, const void* logits,
                   int32_t* argmax, float* conf, bca_stream_t stream);

/*
 * bca_commit_kv -- write finished K/V rows into their pages (a bit copy).
 *
 * "Inference for Interpretable Text-Diffusion Models", "KV Cache", step 3,
 * and "Paged Attention".  For every sequence b and t < num_tokens, row t of
 * k_blk[b] / v_blk[b] ([B, block_size, Hkv, d]; num_tokens <= block_size) is
 * copied to logical position start_pos[b] + t.  Slots not targeted keep
 * their bits.  A target beyond the page table, or a page id outside the pool,
 * is skipped and reported as a device error.
 */
int bca_commit_kv(const bca_dims* dims, const void* k_blk, const void* v_blk, void* k_pool,
                  void* v_pool, const int32_t* page_table, const int32_t* start_pos,
                  int32_t num_tokens, void* workspace, size_t workspace_bytes,
                  bca_stream_t stream);

/*
 * bca_prefill -- block-causal attention over whole prompts, plus the page
 * write of their K/V.
 *
 * "Inference for Interpretable Text-Diffusion Models", "KV Cache", step 1 and
 * the prefill BlockMask figure: P0 = 0, every token attends its own block
 * bidirectionally and earlier blocks causally.  Tiles of 128 queries x 128
 * keys are classified as fully included (no mask), partially included
 * (elementwise mask) or fully excluded (never loaded) ("FlexAttention with
 * Aligned Tiles"); with D = 64 each diagonal tile is partial (3/4 visible).
 *
 * Packed layout: q/out [total_tokens, Hq, d], k/v [total_tokens, Hkv, d];
 * sequence b occupies rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (int32 [B+1],
 * device).  max_seqlen: a host-side upper bound of the sequence lengths.
 * If k_pool is non-NULL, every token t of sequence b is also written to
 * logical position t of b's pages (the cache fill of step 1).
 */
int bca_prefill(const bca_dims* dims, const void* q, const void* k, const void* v,
                const int32_t* cu_seqlens, int32_t total_tokens, int32_t max_seqlen,
                void* k_pool, void* v_pool, const int32_t* page_table, void* out,
                void* workspace, size_t workspace_bytes, bca_stream_t stream);

/*
 * bca_multicanvas -- multi-canvas shrinking-window attention over an arena.
 *
 * "Inference: Fewer, smaller forwards", "Advancement 1", "Advancement 9",
 * "Advancement 11", "Advancement 13".  dims->block_size is the canvas
 * length C; P0 = prompt_len.  The queries of sequence b are its live rows:
 * q_live[b][r] for r < live_count[b], at absolute position live_pos[b][r]
 * (the active-position index list).  A live row of canvas c sees every key
 * whose position is below prompt_len + C*(c+1): arena entries (pages of the
 * pools, the first arena_len[b] slots of b's page list, each with its stored
 * absolute position kv_pos[page][slot]) and live rows (k_live/v_live at
 * live_pos).  Every position must be stored exactly once, in the arena or as
 * a live row; storage order does not matter ("Advancement 10").
 *
 * After the attention, rows commit_rows[b][i] (i < commit_count[b], indices
 * into the live rows) are appended to the arena at slots arena_len[b] + i,
 * with their positions written to kv_pos, and arena_len[b] is increased by
 * commit_count[b] ("Advancement 11": promotion appends at the arena end).
 * commit_rows may be NULL (no promotion).
 *
 * q_live/out [B, max_live, Hq, d]; k_live/v_live [B, max_live, Hkv, d];
 * live_pos int32 [B, max_live] (NULL: row r is at prompt_len + r);
 * live_count int32 [B] (NULL: max_live); kv_pos int32 [num_pages, S];
 * arena_len int32 [B]; commit_rows int32 [B, max_commit]; commit_count [B].
 */
int bca_multicanvas(const bca_dims* dims, const void* q_live, const void* k_live,
                    const void* v_live, const int32_t* live_pos, const int32_t* live_count,
                    int32_t max_live, int32_t prompt_len, int32_t n_canvas, void* k_pool,
                    void* v_pool, const int32_t* page_table, int32_t* kv_pos,
                    int32_t* arena_len, const int32_t* commit_rows,
                    const int32_t* commit_count, int32_t max_commit, void* out,
                    void* workspace, size_t workspace_bytes, bca_stream_t stream);

/*
 * bca_multicanvas_window -- bca_multicanvas for a sliding-window layer.
 *
 * "Inference: Fewer, smaller forwards", "Advancement 11": the arena keeps
 * each entry's absolute position, so a sliding-window attention layer can
 * band-mask the entries that fall outside its window (1024 tokens in the
 * pages' model), which lets up to 5 canvases run even when the prompt plus
 * all canvases exceed the window.  A live row at position q sees a key at
 * position k iff the bca_multicanvas rule holds and q - k < window (the
 * window holds the `window` most recent positions up to q; later keys of
 * the row's own canvas stay visible).  window = 0 is bca_multicanvas;
 * window < 0 is BCA_ERR_INVALID_ARG.  All other arguments as bca_multicanvas.
 */
int bca_multicanvas_window(const bca_dims* dims, const void* q_live, const void* k_live,
                           const void* v_live, const int32_t* live_pos,
                           const int32_t* live_count, int32_t max_live, int32_t prompt_len,
                           int32_t n_canvas, int32_t window, void* k_pool, void* v_pool,
                           const int32_t* page_table, int32_t* kv_pos, int32_t* arena_len,
                           const int32_t* commit_rows, const int32_t* commit_count,
                           int32_t max_commit, void* out, void* workspace,
                           size_t workspace_bytes, bca_stream_t stream);

/*
 * bca_validate_page_table -- host-side debug check of a page table (HOST
 * pointers), for use outside the timed path ("Paged Attention": the page
 * table is used with stricter error checking).  For each sequence b the first
 * ceil(used_tokens[b] / page_size) entries must lie in [0, num_pages) and no
 * page may appear twice among all sequences' used entries.  On failure the
 * offending (sequence, entry) is written to bad_seq/bad_entry (if non-NULL).
 */
int bca_validate_page_table(const bca_dims* dims, const int32_t* page_table_host,
                            const int32_t* used_tokens_host, int32_t* bad_seq,
                            int32_t* bad_entry);

/*
 * bca_decode_static_scratch -- bca_decode for callers that cannot allocate.
 *
 * The pages describe no counterpart to this call; it is a library-side
 * convenience.  It computes exactly what bca_decode computes (same inputs,
 * outputs and commit), but takes no workspace: its scratch is a fixed 16 MiB
 * device array inside the library, present on every GPU that loads the
 * library until the process exits.  It is meant for callers that must not
 * call cudaMalloc on this path: a plugin inside an engine that owns all
 * device memory and offers it no allocator, a serving loop in which an
 * allocation (which can synchronize the device or fail under fragmentation)
 * is not acceptable, or a runtime with no access to the CUDA allocator.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *  - A request whose minimum decode scratch exceeds the array
 *    (bca_workspace_size(dims, BCA_OP_DECODE_MIN) > 16 MiB) is rejected with
 *    BCA_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.
 *  - Every call shares the one array and it keeps the last call's contents:
 *    the status header is cleared at the start of each call, and calls that
 *    overlap on the GPU (other streams, other host threads) race on it.
 *  - device_status: optional device int32 that receives, in stream order, the
 *    first device-detected error of this call (0 if none).
 */
int bca_decode_static_scratch(const bca_dims* dims, const void* q, const void* k_blk,
                              const void* v_blk, void* k_pool, void* v_pool,
                              const int32_t* page_table, const int32_t* prefix_len, void* out,
                              int commit, int32_t* device_status, bca_stream_t stream);

/*
 * Kernel timing for benchmarks (not on any computation path).  While a
 * profile is active, every entry point records a CUDA event pair around each
 * kernel it launches, on the call's own stream; bca_profile_stop synchronizes
 * those events and returns, per kernel kind, the number of launches and their
 * summed device time.  Host-side state, one profile per process; the event
 * pairs are created by bca_profile_start (max_launches of them) and destroyed
 * by bca_profile_stop.  Launches beyond max_launches are not timed.  Do not
 * use while a stream is being captured into a CUDA graph.
 */
#define BCA_KERNEL_ATTENTION 0 /* the block-causal attention kernel */
#define BCA_KERNEL_COMBINE 1   /* decode epilogue: KV commit and split-KV combine */
#define BCA_KERNEL_COMMIT 2    /* KV commit / prefill page write */
#define BCA_KERNEL_PROMOTE 3   /* multicanvas arena promotion */
#define BCA_KERNEL_PLAN 4      /* work planning (prefill, multicanvas, decode batches > 64) */
#define BCA_KERNEL_CONFIDENCE 5 /* softmax-plus-argmax over the vocabulary */
#define BCA_KERNEL_QKV_POST 6  /* norms + RoPE + cache write after the QKV projection */
#define BCA_KERNEL_KINDS 7

typedef struct bca_kernel_times {
  int32_t launches[BCA_KERNEL_KINDS];
  double total_ms[BCA_KERNEL_KINDS];
} bca_kernel_times;

int bca_profile_start(int32_t max_launches);
int bca_profile_stop(bca_kernel_times* out);

#ifdef __cplusplus
}
#endif

#endif /* BCA_H_ */
