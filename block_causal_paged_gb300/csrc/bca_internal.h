// Internal declarations shared by the host API and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

struct bca_dims;  // the public call dimensions (bca.h)

namespace bca {

constexpr int kTileKeys = 128;    // keys per KV tile
constexpr int kChunkKeys = 16;    // keys per TMA box (a page holds whole chunks)
constexpr int kChunksPerTile = kTileKeys / kChunkKeys;
constexpr int kRowsPerMTile = 128;
constexpr int kThreads = 384;     // 12 warps, see the role map in attention.cu
constexpr int kFusedPlanMax = 64; // decode batches up to this are planned inside the attention kernel
constexpr int kMaxDevices = 64;   // per-device launch caches (device ordinals beyond: no cache)
// Per internal wait: about 2 s at the maximum SM clock (longer when clocked down).
constexpr long long kWaitTimeoutCycles = 4000000000ll;

enum Mode : int { kModeDecode = 0, kModePrefill = 1, kModeMulticanvas = 2 };

// First 256 bytes of every workspace.
struct WsHeader {
  int32_t status;          // first device-detected error (0 = none)
  int32_t chunk_tiles;     // decode: KV tiles per split chunk chosen by the plan kernel
  int32_t n_items;         // work items of the current call
  int32_t work_next;       // next work item to hand out (reset by the plan kernel)
  unsigned long long tiles_full;
  unsigned long long tiles_partial;
  unsigned long long tiles_skipped;
  int32_t n_split_slots;   // decode: split-KV slots in use (plan)
  int32_t exit_count;      // attention CTAs finished in the current launch (reset by the last)
  // the first internal wait that timed out: 1 once recorded, the CTA, the warp,
  // the barrier's byte offset in the CTA's shared memory and the awaited parity
  int32_t wait_fail[5];
  int32_t reserved1[47];
};
static_assert(sizeof(WsHeader) == 256, "header size");
constexpr size_t kWsHeaderBytes = 256;

// Decode workspace: header | split_base int32[B] | item list int4[2][items_cap]
// | slot table int4[cap] | partial (max, sum) float2[cap][256] | partial O
// float[cap][d/4][256][4] (regions 256-byte aligned).  items_cap bounds the
// number of work items (n_sms * waves + B * Hkv * n_rb); cap (split-KV slots)
// is whatever fits.
struct DecodeWsLayout {
  size_t split_base_off, items_off, slot_off, ml_off, o_off, bytes_per_slot;
  int items_cap;
  int cap;
};
DecodeWsLayout decode_ws_layout(int B, int Hkv, int n_rb, int head_dim, int n_sms, size_t ws_bytes);
size_t decode_ws_recommended(int B, int Hkv, int n_rb, int head_dim, int n_sms);
size_t decode_ws_minimum(int B, int Hkv, int n_rb, int head_dim, int n_sms);

struct AttnParams {
  int mode;
  int B, Hq, Hkv, G, S, num_pages, max_pages;
  int Dblk;            // decode/prefill block size D, or canvas length C
  int hpr, tpm;        // heads per row group and tokens per M-tile (hpr * tpm <= 128)
  int n_hp;            // prefill: M-tile pairs (heads) per KV head
  int n_rb;            // decode: row blocks per KV head (each = 2 M-tiles)
  int ch_min, waves;   // decode split policy
  int fused_plan;      // decode: every CTA plans for itself (batch <= kFusedPlanMax)
  int pair;            // launched on CTA pairs (attention_pair.cu): one work unit per pair
  int causal;          // decode: the D query tokens attend each other causally (short
                       // extend; the prefix length then need not be a multiple of D)
  int n_qt_max;        // prefill: query tiles of the longest sequence (host bound)
  int n_rb_max;        // multicanvas: row blocks of the longest live list (host bound)
  float scale_log2;    // softmax scale * log2(e)
  const int32_t* page_table;
  const int32_t* lens;       // decode prefix_len | prefill cu_seqlens | multicanvas live_count
  const int32_t* live_pos;   // multicanvas (may be null)
  const int32_t* kv_pos;     // multicanvas arena positions [num_pages, S]
  const int32_t* arena_len;  // multicanvas
  int max_live, prompt_len;
  int window;                // multicanvas: sliding-window band (key kept iff q - k < window); 0: none
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const uint16_t* k_dense;   // decode k_blk | prefill k | multicanvas k_live
  const uint16_t* v_dense;
  int pool_rows;             // num_pages * Hkv * S
  int dense_tokens;          // token rows of the dense K/V view
  uint16_t* out;             // bf16 [q_tokens, Hq, d]
  int out_align32;           // out is 32-byte aligned: the pair kernel stores 32 bytes at a time
  WsHeader* hdr;
  int32_t* split_base;
  int4* items;               // decode: item list written by the plan kernel
  int items_cap;
  int4* slot_info;           // decode: per split slot {b, g << 16 | rb, first slot of its group, chunks}
  float* part_ml;
  float* part_o;
  int split_cap;
  // decode with commit: the block's K/V (k_dense / v_dense) is copied into
  // these pools by the decode epilogue kernel, after the attention kernel
  // (null: no commit)
  uint16_t* commit_k;
  uint16_t* commit_v;
  // multicanvas: {smallest, largest} key position of arena tile a of sequence
  // b at tile_kv[b * n_at_max + a], written by the plan kernel
  int2* tile_kv;
  int n_at_max;              // arena tiles per sequence: ceil(max_pages * S / 128)
};

// Multicanvas workspace: header | arena tile summaries int2[B][n_at_max].
size_t multicanvas_ws_bytes(int B, int max_pages, int S);

struct AttnMaps {
  CUtensorMap q, kp, vp, kd, vd;
};

// Plan kernel: resets the work counter; for decode also chooses the split
// chunk, orders sequences longest first and writes the item list; for
// multicanvas summarizes the key positions of every arena tile.
cudaError_t launch_plan(const AttnParams& p, int attn_grid, cudaStream_t stream);

// Launch the block-causal attention kernel (decode, prefill or multicanvas).
cudaError_t launch_attention(const AttnParams& p, const AttnMaps& maps, int head_dim, int grid,
                             cudaStream_t stream);

// Launch the CTA-pair attention kernel (decode or extend with two M-tiles in
// the first row block, prefill, multicanvas; head_dim 128) on n_pairs
// clusters of two CTAs.
cudaError_t launch_attention_pair(const AttnParams& p, const AttnMaps& maps, int n_pairs,
                                  cudaStream_t stream);
// Clusters of two CTAs of that kernel that can be resident at once (0 on error).
int attention_pair_max_pairs(int n_sms);

// Split-KV combine for decode: one CTA per (split group, 32 head-dim columns),
// over the slot table the plan kernel wrote.
cudaError_t launch_decode_combine(const AttnParams& p, int head_dim, int n_sms, cudaStream_t stream);

// Softmax-plus-argmax over the vocabulary (dtype 0: bf16, 1: fp32).
cudaError_t launch_confidence(int64_t rows, int vocab, int64_t ld, int dtype, const void* logits,
                              int32_t* argmax, float* conf, cudaStream_t stream);

// Bit copy of K/V rows into pages.  Source rows are [rows, Hkv, d]; sequence
// b owns rows src_first(b) .. src_first(b)+count(b)-1 and writes them to
// logical positions start(b) .. start(b)+count(b)-1 of its pages.
//   cu != null (prefill): src_first = cu[b], count = cu[b+1]-cu[b], start = 0
//   cu == null (commit):  src_first = b*rows_per_seq, count = num_tokens,
//                         start = start_pos[b]
struct CommitParams {
  const uint16_t* k_src;
  const uint16_t* v_src;
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* page_table;
  const int32_t* start_pos;
  const int32_t* cu;
  int rows_per_seq;
  int num_tokens;
  int max_rows;                 // host bound on count(b), for the grid
  int B, Hkv, d, S, num_pages, max_pages;
  WsHeader* hdr;
};
cudaError_t launch_commit(const CommitParams& c, cudaStream_t stream);

// QKV-post: norms + RoPE of the projection's output, optional cache write.
struct QkvPostParams {
  const uint16_t* qkv;        // [B * n, Hq + 2 Hkv, d]
  const int32_t* positions;   // [B * n] (may be null without RoPE / kv_pos)
  const uint16_t* q_norm_w;   // [d] or null
  const uint16_t* k_norm_w;   // [d] or null
  float eps, rope_theta;      // rope_theta 0: no rotation
  // RoPE frequency of pair i (< d/2) in turns per position, as a 64-bit
  // fixed-point fraction: round(theta^(-2i/d) / (2 pi) * 2^64)
  unsigned long long rope_turns[64];
  uint16_t* q_out;            // [B * n, Hq, d]
  uint16_t* k_out;            // [B * n, Hkv, d]
  uint16_t* v_out;
  const int32_t* write_pos;   // [B * n] cache position, -1 = none; null: no cache write
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* page_table;
  int32_t* kv_pos;            // [num_pages, S] or null
  int B, n, Hq, Hkv, S, num_pages, max_pages;
  WsHeader* hdr;
};
cudaError_t launch_qkv_post(const QkvPostParams& c, int head_dim, int n_sms, cudaStream_t stream);

// Arena promotion after a multicanvas step.
struct PromoteParams {
  const uint16_t* k_live;
  const uint16_t* v_live;
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* page_table;
  const int32_t* live_pos;
  const int32_t* live_count;
  int32_t* kv_pos;
  int32_t* arena_len;
  const int32_t* commit_rows;
  const int32_t* commit_count;
  int B, Hkv, d, S, num_pages, max_pages, max_live, max_commit, prompt_len;
  WsHeader* hdr;
};
cudaError_t launch_promote(const PromoteParams& c, cudaStream_t stream);

// Host-side input checks for BCA_DEBUG=1 (debug_check.cu): lengths,
// positions and page-table entries copied to the host and checked before a
// launch; BCA_OK or the error the entry point returns.
bool debug_enabled();
int debug_check_decode(const bca_dims* d, const int32_t* page_table,
                       const int32_t* prefix_len, int commit, int causal, cudaStream_t s);
int debug_check_prefill(const bca_dims* d, const int32_t* cu_seqlens, int32_t total_tokens,
                        int32_t max_seqlen, const int32_t* page_table, cudaStream_t s);
int debug_check_commit(const bca_dims* d, const int32_t* page_table,
                       const int32_t* start_pos, int32_t num_tokens, cudaStream_t s);
int debug_check_qkv_post(const bca_dims* d, const int32_t* write_pos,
                         const int32_t* page_table, cudaStream_t s);
int debug_check_multicanvas(const bca_dims* d, const int32_t* live_count, int32_t max_live,
                            const int32_t* page_table, const int32_t* arena_len,
                            const int32_t* commit_rows, const int32_t* commit_count,
                            int32_t max_commit, cudaStream_t s);

}  // namespace bca
