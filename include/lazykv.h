/*
 * lazykv.h -- C ABI of liblazykv.so: LazyAttention's hot path on one GB300 (sm_103a).
 *
 * LazyAttention ("LazyAttention: Efficient Retrieval-Augmented Generation with Deferred
 * Positional Encoding", ICML 2026) keeps ONE position-free KV copy per document and applies
 * the positional encoding inside the attention kernels.  Sources cited below:
 *   [NOTE]   papernotes.org reading note on the paper: sections 方法详解/整体框架
 *            (position-free cache, Example 3.1), 关键设计 (Deferred Positional Encoding;
 *            Tiling 感知的 Q/K 旋转分派; 融合 Triton kernel + bit-packed 元数据), 通用性.
 *   [GIST]   gist.science technical summary: Implementazione Tecnica (Prefilling,
 *            Decoding), Equivalenza Matematica.
 *   [README] illinoisdata/lazy-attention README mirror: Variants (scheduler metadata).
 *
 * Conventions for every entry point
 *   - Pointers marked (host) are CPU memory; (device) are GPU memory the CALLER allocated
 *     (e.g. by PyTorch) and owns.  The library allocates no device memory and keeps no state
 *     beyond one 32-bit device status word per GPU (see lazy_device_status).
 *   - bf16 tensors are contiguous, row-major, 16-byte aligned.
 *   - Paged caches: k_cache and v_cache are bf16 [num_pages][Hkv][16][D]; one page of one KV
 *     head is 16 * D * 2 bytes, contiguous.  A cache slot is page * 16 + row.  The attention
 *     kernels read only rows that hold a key the query can see (a block's first n_valid rows,
 *     and in the query segment none past the query's position), so the rest of a page may hold
 *     anything, uninitialised or NaN bits included.
 *   - Every GPU entry point is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream), performs no synchronisation and returns after the launch.
 *   - Kernels are launched with programmatic dependent launch: one may become resident while
 *     the previous kernel of the stream drains, and it reads or writes no global memory until
 *     that kernel has completed (griddepcontrol.wait), so stream order is kept exactly as for
 *     a plain launch, including inside CUDA graph capture.
 *   - Return codes: LAZY_OK, or a negative code with a message for lazy_last_error().
 *     Argument errors are detected on the host before anything is launched.  Errors found
 *     by a kernel (an out-of-range page or slot, a wait that ran out) set bits of the device
 *     status word and the offending element is skipped; no kernel traps or asserts.
 *   - Head dims supported: D in {64, 128}; rotary_dim a multiple of 16 in [16, D] (RoPE and
 *     YaRN).  Hq % Hkv == 0.
 */
#ifndef LAZYKV_H
#define LAZYKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LAZY_OK 0
#define LAZY_EINVAL (-1) /* shape, pointer, alignment or dtype argument not supported     */
#define LAZY_ERANGE (-2) /* a value does not fit a field of the 64-bit block word, or max_blocks too small */
#define LAZY_ECUDA (-3)  /* a CUDA runtime call or kernel launch failed                   */
#define LAZY_EARCH (-4)  /* the current GPU is not compute capability 10.x                */
#define LAZY_EDEVICE (-5) /* a kernel reported an error through the device status word    */

#define LAZY_PAGE_SIZE 16

/* Device status word bits (lazy_device_status). */
#define LAZY_STATUS_BAD_PAGE 1u    /* a block word named a page >= num_pages            */
#define LAZY_STATUS_BAD_SLOT 2u    /* kv_write got a slot outside the caches             */
#define LAZY_STATUS_TIMEOUT 4u     /* a bounded wait on a copy or MMA ran out            */
#define LAZY_STATUS_BAD_ROW 8u     /* a query row's visible range exceeded max_blocks    */

/* Positional encodings ([NOTE] 通用性: RoPE variants and ALiBi change only metadata). */
enum {
  LAZY_POS_ROPE = 0,  /* RoPE, theta_i = rope_theta^(-2i/rotary_dim); half-split pairs
                         (x_i, x_{i+rotary_dim/2}) or interleaved (x_2i, x_2i+1)          */
  LAZY_POS_YARN = 1,  /* YaRN-scaled RoPE frequencies (YaRN paper's ramp) + mscale^2     */
  LAZY_POS_ALIBI = 2, /* no rotation; logit += -alibi_slopes[h] * (m - p)                */
  LAZY_POS_NONE = 3   /* no positional work at all: the "Delta = 0" twin used to time the
                         cost of deferred rotation (same kernels, rotation compiled out)  */
};

/*
 * Positional configuration, read on the host at call time (by value semantics).
 *   rope_theta, rotary_dim          RoPE base and rotated width: the first rotary_dim
 *                                   dimensions of every head are rotated, the rest pass
 *                                   through (a multiple of 16 in [16, D]).
 *   yarn_factor, yarn_orig_ctx,     YaRN scale s, original context L0, ramp bounds
 *   yarn_beta_fast, yarn_beta_slow  (defaults 32 and 1 when given as 0).
 *   alibi_slopes                    (device) float [Hq]; ALiBi only.
 *   cos_sin                         (device) float [max_pos][rotary_dim] table written by
 *                                   lazy_build_rope_table (cos in the first half of a row,
 *                                   sin in the second), or NULL: compute cos/sin on the fly.
 *   max_pos                         rows of cos_sin.
 *   interleaved                     0: half-split pairs (x_i, x_{i + rotary_dim/2}) (NeoX /
 *                                   Llama); 1: adjacent pairs (x_2i, x_2i+1) (GPT-J).  The
 *                                   pages treat RoPE variants as metadata ([NOTE] 通用性).
 */
typedef struct lazy_pos_cfg {
  int32_t kind;
  int32_t rotary_dim;
  float rope_theta;
  float yarn_factor;
  int32_t yarn_orig_ctx;
  float yarn_beta_fast;
  float yarn_beta_slow;
  const float* alibi_slopes;
  const float* cos_sin;
  int32_t max_pos;
  int32_t interleaved;
} lazy_pos_cfg;

/*
 * lazy_build_doc_meta -- per-request block list with one packed 64-bit word per block.
 * [README] Variants (the scheduler builds rotation metadata); [NOTE] 融合 Triton kernel +
 * bit-packed 元数据 (block id, offset and mask in one 64-bit register); [NOTE] 整体框架
 * (each document indexed from local position 0; the request places it at offset Delta).
 *
 * All pointers (host).  Request b lists documents req_docs[req_doc_off[b] .. req_doc_off[b+1]),
 * each an index into doc_len [n_docs] and the page lists doc_pages[doc_page_off[d] ..
 * doc_page_off[d+1]).  Its query segment (prefill tokens then decode tokens) has q_len[b]
 * prefill tokens and capacity pages q_pages[q_page_off[b] .. q_page_off[b+1]).
 * Outputs, each [B][max_blocks] or [B], fully written (unused tail entries = 0):
 *   block_table  int32  physical page of each block
 *   meta         uint64 word: bits [4:0] n_valid (1..16), [15:5] page index within the
 *                document pg (< 2048), [39:16] Delta (< 2^24), [63:40] physical page (< 2^24).
 *                Key row t of a block sits at absolute position p = Delta + 16 * pg + t.
 *                Query-segment blocks are listed as full (n_valid = 16); causality (p <= m)
 *                masks their unwritten rows, and the attention kernels never read them.
 *   seq_len      keys visible after the prefill tokens are written (= q_start + q_len)
 *   q_start      Delta of the query segment (= total document length)
 *   doc_blocks   number of document blocks (the query segment starts at this block)
 * Returns LAZY_EINVAL for negative lengths or missing pages, LAZY_ERANGE when a field
 * overflows or a request needs more than max_blocks blocks.  Deterministic, bit-exact.
 */
int lazy_build_doc_meta(int B, const int32_t* req_doc_off, const int32_t* req_docs, int n_docs,
                        const int32_t* doc_len, const int32_t* doc_page_off,
                        const int32_t* doc_pages, const int32_t* q_len,
                        const int32_t* q_page_off, const int32_t* q_pages, int max_blocks,
                        int32_t* block_table, uint64_t* meta, int32_t* seq_len,
                        int32_t* q_start, int32_t* doc_blocks);

/*
 * lazy_build_rope_table -- cos/sin table for the positional config ([NOTE] Tiling 感知:
 * cos/sin read from a table, one D-length vector per document offset).
 * out_table (device) float [max_pos][rotary_dim]: row p holds cos(p theta_i) for i < d/2,
 * then sin(p theta_i).  Angles are reduced exactly (fixed-point turn count), so row p is
 * accurate to ~2e-7 for every p < 2^24.  ALiBi / NONE: LAZY_EINVAL.
 */
int lazy_build_rope_table(const lazy_pos_cfg* cfg, int max_pos, float* out_table, void* stream);

/*
 * lazy_kv_write -- write T tokens into the paged caches, position-free ([NOTE] 整体框架:
 * the cache holds content indexed from each document's local position 0).
 *   k, v       (device) bf16 [T][Hkv][D], raw (pre-RoPE) keys and values
 *   slot       (device) int32 [T], page * 16 + row of each token
 *   local_pos  (device) int32 [T], position j of the token inside its document / segment
 * Stored K = bf16_RNE(R_j k) computed in fp32 (RoPE/YaRN); raw k for ALiBi/NONE.
 * Stored V = v.  A slot outside [0, num_pages * 16) sets LAZY_STATUS_BAD_SLOT and the token
 * is skipped.
 */
int lazy_kv_write(const void* k, const void* v, const int32_t* slot, const int32_t* local_pos,
                  int T, int Hkv, int D, void* k_cache, void* v_cache, int num_pages,
                  const lazy_pos_cfg* cfg, void* stream);

/*
 * lazy_attn_decode -- one decode step (M = 1 per request), GQA-grouped, split over the KV
 * sequence.  [NOTE] Tiling 感知的 Q/K 旋转分派: decode rotates Q, and only when the KV block
 * crosses a document boundary; [NOTE] 融合 Triton kernel: the block word is unpacked from a
 * register; [GIST] Decoding.
 *   q          (device) bf16 [B][Hq][D] raw queries; request b's query sits at
 *              m = seq_len[b] - 1 and its own key/value were written at p = m beforehand
 *   seq_len, q_start, doc_blocks  (device) int32 [B] from lazy_build_doc_meta (seq_len
 *              advanced by the caller for every decode token written)
 *   meta       (device) uint64 [B][max_blocks]
 *   scale      softmax scale; 0 selects 1/sqrt(D) (times mscale^2 for YaRN)
 *   out        (device) bf16 [B][Hq][D];  lse (device, nullable) float [B][Hq], natural log
 *   ws         (device) workspace of at least lazy_workspace_size(LAZY_PHASE_DECODE, ...)
 *              bytes, 256-byte aligned, or NULL when that size is 0.
 * Keys visible to m: every document block plus the query segment up to p <= m.
 */
int lazy_attn_decode(const void* q, const int32_t* seq_len, const int32_t* q_start,
                     const int32_t* doc_blocks, const uint64_t* meta, int B, int max_blocks,
                     const void* k_cache, const void* v_cache, int num_pages, int Hq, int Hkv,
                     int D, float scale, const lazy_pos_cfg* cfg, void* out, float* lse,
                     void* ws, size_t ws_bytes, void* stream);

/*
 * lazy_attn_decode_noalloc -- lazy_attn_decode for callers that cannot allocate device memory.
 * The paper has no counterpart: this is a deployment variant of the decode above.
 *
 * Who needs it: a host that owns all GPU memory itself (e.g. an engine that reserves HBM for
 * its KV pool at start-up and gives plugins no allocator), or a latency-bound loop that must
 * never call cudaMalloc (which can synchronise the device).  Such callers cannot pass the
 * split-KV workspace lazy_attn_decode needs, so this entry point uses a fixed 16 MiB array
 * compiled into the library instead; neither the caller nor the library allocates (no
 * cudaMalloc, cudaFree or allocating library routine is called).
 *   Arguments, layouts and results: exactly those of lazy_attn_decode, without ws/ws_bytes.
 *   Limit: batches whose split scratch (see lazy_workspace_size) exceeds 16 MiB are rejected
 *          with LAZY_EINVAL and a message; nothing is launched.
 *   Memory: every GPU that loads the library holds the 16 MiB array until the process exits.
 *   Set-up: the first call on each device looks up the array's device address (with that
 *          device current); make that first call before any stream capture.
 *   Sharing: all calls on a device share the one array and it keeps the last call's contents.
 *          Nothing in it must start at zero.  Calls that overlap on the GPU (different
 *          streams, or different host threads) race on it: serialise them.
 */
int lazy_attn_decode_noalloc(const void* q, const int32_t* seq_len, const int32_t* q_start,
                             const int32_t* doc_blocks, const uint64_t* meta, int B,
                             int max_blocks, const void* k_cache, const void* v_cache,
                             int num_pages, int Hq, int Hkv, int D, float scale,
                             const lazy_pos_cfg* cfg, void* out, float* lse, void* stream);

/*
 * lazy_attn_prefill -- causal prefill of every request's query tokens over its documents and
 * its own earlier tokens.  [NOTE] Tiling 感知: prefill rotates each K tile by its document's
 * Delta (Q tiles are much taller than K tiles); [NOTE] 融合 Triton kernel (K tile split in
 * halves, rotated per half-dimension, then the GEMM); [GIST] Prefilling.
 *   q          (device) bf16 [total_q][Hq][D] raw queries; rows cu_q[b] .. cu_q[b+1] belong
 *              to request b and sit at absolute positions q_start[b] + i.  Their keys and
 *              values must already be in the cache (lazy_kv_write with local_pos = i).
 *   cu_q       (device) int32 [B+1];  max_q = max_b (cu_q[b+1] - cu_q[b]) (host value)
 *   out        (device) bf16 [total_q][Hq][D];  lse (device, nullable) float [total_q][Hq]
 *   ws / ws_bytes as for decode, sized by lazy_workspace_size(LAZY_PHASE_PREFILL, ...).
 */
int lazy_attn_prefill(const void* q, const int32_t* cu_q, const int32_t* q_start,
                      const int32_t* doc_blocks, const uint64_t* meta, int B, int max_blocks,
                      int total_q, int max_q, const void* k_cache, const void* v_cache,
                      int num_pages, int Hq, int Hkv, int D, float scale,
                      const lazy_pos_cfg* cfg, void* out, float* lse, void* ws,
                      size_t ws_bytes, void* stream);

#define LAZY_PHASE_DECODE 0
#define LAZY_PHASE_PREFILL 1

/*
 * lazy_workspace_size -- bytes of workspace the given call needs (0 if none).
 * rows = B for decode, total_q for prefill.  Uses the current device's SM count, so query it
 * with the device that will run the call current.
 */
size_t lazy_workspace_size(int phase, int rows, int B, int max_blocks, int Hq, int Hkv, int D);

/*
 * lazy_device_status -- synchronise `stream`, then read and clear the current device's
 * status word into *status (LAZY_STATUS_* bits; 0 = no kernel reported a problem).
 */
int lazy_device_status(void* stream, uint32_t* status);

/* Thread-local message for the last non-zero return code of this thread. */
const char* lazy_last_error(void);

/* ------------------------------------------------------------------------------------------
 * Document cache manager (host only).  [NOTE] 研究背景与动机 (核心矛盾: with a Zipf document
 * popularity, D possible positions and a budget of C entries, a position-free cache holds the
 * top C documents while a position-aware one holds only floor(C/D) of them) and 关键设计
 * (Deferred Positional Encoding: one physical copy serves every position).
 * Decides which documents' pages are resident in a pool of num_pages pages ([0, num_pages) of
 * the K/V caches).  position_aware = 0: one entry per document (this library's cache);
 * position_aware = 1: one entry per (document, position) variant (the design the pages
 * compare against; for simulation).  Least-recently-used eviction among entries no batch
 * holds.  The handle is host memory owned by the caller (create / destroy); not thread-safe.
 * ------------------------------------------------------------------------------------------ */
typedef struct lazy_doc_cache lazy_doc_cache;
/* NULL on error (num_pages outside [1, 2^24]; lazy_last_error says why). */
lazy_doc_cache* lazy_doc_cache_create(int num_pages, int position_aware);
void lazy_doc_cache_destroy(lazy_doc_cache* cache);
/* Look up without changing recency or pins: returns the entry's page count (its page ids copied
 * to pages_out (host) if not NULL and max_pages is large enough), 0 if not resident, < 0 on an
 * argument error.  `pos` is ignored by a position-agnostic cache. */
int lazy_doc_cache_lookup(lazy_doc_cache* cache, int doc, int pos, int32_t* pages_out, int max_pages);
/* Hold document `doc` (at position `pos`) for a batch: on a hit (*hit = 1) copies its n_pages
 * page ids to pages_out (host); on a miss (*hit = 0) evicts unheld least-recently-used entries
 * until n_pages pages are free and assigns them (the caller then writes the document there, e.g.
 * with lazy_kv_write at local positions).  Either way the entry is pinned until
 * lazy_doc_cache_release.  LAZY_ERANGE if held entries leave no room; LAZY_EINVAL on bad
 * arguments or a cached entry of another size. */
int lazy_doc_cache_acquire(lazy_doc_cache* cache, int doc, int pos, int n_pages, int32_t* pages_out, int* hit);
int lazy_doc_cache_release(lazy_doc_cache* cache, int doc, int pos);
/* Counters since creation (any pointer may be NULL). */
int lazy_doc_cache_stats(const lazy_doc_cache* cache, long long* hits, long long* misses, long long* evictions,
                         int* entries, int* free_pages);

/* Library version, e.g. 100 for 0.1.0. */
int lazy_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LAZYKV_H */
