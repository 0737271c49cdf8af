/*
 * cpattn.h -- C ABI of libcpattn.so: causal GQA partial attention over logical
 * context-parallel (CP) shards on one GB300 (sm_103a), with LSE merge.
 *
 * Sources (vLLM pull-request pages):
 *   [PKV]  "Add utility functions to enable pass-kv prefill and allgather decode"
 *          (PR 26059), Purpose: attention is the only op that couples tokens of a
 *          sequence; in prefill both Q and KV are split over CP ranks and either the
 *          KV shards (full prefill) or the Q shards (chunked prefill with a long
 *          cached context) travel past the resident ones while partial attention
 *          runs; in decode the KV stays round-robin on the ranks, the query is made
 *          available to all of them and their partial results are combined.
 *   [PCP]  "[Feature] Prefill Context Parallel (PCP) basic support" (PR 28718),
 *          Purpose and code-review summary: block tables extended for decode and
 *          prefill CP; one kv-cache interleave size shared by both.
 *   [GQA]  "[Feature] Support Prefill Context Parallel (PCP) for GQA flashinfer"
 *          (PR 28723), Purpose and Test Plan: token partitioning for prefill CP,
 *          GQA attention backend, interleave size 8.
 *
 * All CP ranks are LOGICAL: every shard lives in this GPU's memory and no call
 * communicates with another GPU.
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller allocates and frees every buffer.  Pointers named
 *     "device" must be device memory of the current CUDA device; "host" pointers
 *     are read before the call returns.  The library never allocates, frees or
 *     synchronises; work is enqueued on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and returns immediately.
 *   - Errors: argument errors are detected on the host, nothing is launched and a
 *     non-zero cp_status is returned; cp_last_error() then gives a one-line reason
 *     (thread-local).  A failed launch returns CP_ERR_CUDA.  Conditions only the
 *     device can see (a block-table entry outside the pool, a pipeline wait that
 *     ran out of its iteration budget) are written to the optional device word
 *     `err` (first error wins, CP_OK is never written) and the affected work is
 *     skipped; read it after synchronising the stream.
 *   - Layout: tensors are dense, row-major, in the index order written beside them,
 *     16-byte aligned.  Heads: query head h reads kv head h / (Hq / Hkv).
 *   - LSE values are natural-log log-sum-exp of the scaled scores; an empty key set
 *     gives LSE = -inf and an output row that is never read (see cp_lse_merge).
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CPATTN_ABI_VERSION 3

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or shape          */
  CP_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, dtype, block size     */
  CP_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed                 */
  CP_ERR_TIMEOUT = 4,       /* device: a pipeline wait exceeded its budget          */
  CP_ERR_DEVICE_BOUNDS = 5  /* device: an index (page id, position) out of range    */
} cp_status;

typedef enum { CP_F32 = 0, CP_BF16 = 1 } cp_dtype;
typedef enum { CP_PASS_KV = 0, CP_PASS_Q = 1 } cp_mode;
typedef enum {
  CP_IMPL_AUTO = 0,     /* tcgen05 tensor-core kernel for bf16, SIMT kernel for f32   */
  CP_IMPL_TCGEN05 = 1,  /* bf16 only: TMA + tcgen05.mma + TMEM                        */
  CP_IMPL_SIMT = 2,     /* plain CUDA cores, any supported dtype (cross-check path)   */
  CP_IMPL_TCGEN05_SINGLE = 3  /* bf16: tcgen05 kernel with one q head per CTA (the     */
                              /* default pairs two heads, or two row tiles of one head */
                              /* when q heads per kv head is odd)                      */
} cp_impl;

/* Human-readable name of a cp_status value (static string). */
const char* cp_status_string(int32_t status);

/* Copies the reason for the calling thread's last failed call into buf (NUL-
 * terminated, truncated to n bytes) and returns that call's status. */
int32_t cp_last_error(char* buf, size_t n);
/* The same call under its longer name. */
int32_t cp_last_error_detail(char* buf, size_t n);

/* CPATTN_ABI_VERSION of the loaded library. */
int32_t cp_abi_version(void);

/* ------------------------------------------------------------------------------
 * cp_partition -- load-balanced token partition for prefill CP ([GQA] Purpose:
 * token partitioning; [PKV] Purpose: Q and KV both sharded in prefill).
 *
 * Each sequence of T tokens is cut into 2*cp chunks with bounds
 * b_k = floor(k*T/(2*cp)); logical rank r holds chunk r then chunk 2cp-1-r.
 * Shard-major order lists rank 0's rows first (sequence by sequence, chunk r
 * before chunk 2cp-1-r), then rank 1's, and so on.
 *
 *   cu_seqlens    device int32 [num_seqs+1], cu_seqlens[0] = 0, non-decreasing,
 *                 cu_seqlens[num_seqs] = total_tokens (rows beyond total_tokens are
 *                 not written).
 *   perm          device int32 [total_tokens] or NULL: shard-major row -> token.
 *   inv_perm      device int32 [total_tokens] or NULL: token -> shard-major row.
 *   shard_offsets device int32 [cp+1] or NULL: first shard-major row of each rank.
 *   chunk_bounds  device int32 [num_seqs][2cp+1] or NULL: b_k within each sequence.
 * Requires 1 <= cp <= 64 and num_seqs*cp <= 16384.  Bit-exact integer output.
 * ---------------------------------------------------------------------------- */
cp_status cp_partition(const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                       int32_t cp, int32_t* perm, int32_t* inv_perm, int32_t* shard_offsets,
                       int32_t* chunk_bounds, void* stream);

/* ------------------------------------------------------------------------------
 * cp_kv_interleave_layout -- round-robin kv placement ([PKV] Purpose: decode KV
 * stored round-robin on the CP ranks; [PCP] code-review summary: interleave size
 * shared by prefill and decode CP; [PCP] Purpose: block tables per CP rank).
 *
 * Position p of a sequence goes to rank rho = floor(p/I) mod cp at local index
 * l = floor(p/(I*cp))*I + p mod I (groups of I positions dealt in turn, each rank
 * keeping arrival order).  Rank r holds
 * L_r = floor(L/(I*cp))*I + clamp(L mod (I*cp) - r*I, 0, I) tokens of a length-L
 * sequence.  The slot of a token in its rank's page pool is
 * block_tables[rho][b][l / block_size] * block_size + l mod block_size.
 *
 *   cu_seq_lens    device int32 [num_seqs+1] prefix sums of sequence lengths.
 *   block_tables   device int32 [cp][num_seqs][max_blocks] (needed for slots only).
 *   local_lens     device int32 [cp][num_seqs] or NULL.
 *   rank_of_token  device int32 [total_tokens] or NULL.
 *   local_of_token device int32 [total_tokens] or NULL.
 *   slot_of_token  device int64 [total_tokens] or NULL (needs block_tables).
 *   err            device int32 or NULL: CP_ERR_DEVICE_BOUNDS if a slot needs a
 *                  table column >= max_blocks or a negative page id (slot = -1).
 * Bit-exact integer output.
 * ---------------------------------------------------------------------------- */
cp_status cp_kv_interleave_layout(const int32_t* cu_seq_lens, int32_t num_seqs,
                                  int32_t total_tokens, int32_t cp, int32_t interleave,
                                  int32_t block_size, const int32_t* block_tables,
                                  int32_t max_blocks, int32_t* local_lens, int32_t* rank_of_token,
                                  int32_t* local_of_token, int64_t* slot_of_token, int32_t* err,
                                  void* stream);

/* ------------------------------------------------------------------------------
 * cp_kv_cache_write -- store new tokens' K/V into the per-rank paged pools at their
 * round-robin slots ([PKV] Purpose: KV kept round-robin on the CP ranks; [PCP] Purpose:
 * per-rank block tables; [PCP] code-review summary: one interleave size for PCP and DCP).
 *
 * Sequence b's new rows cu_new[b] .. cu_new[b+1]-1 of k_new / v_new ([N][Hkv][d], token-major)
 * hold positions start_pos[b], start_pos[b]+1, ...; each row goes to rank
 * rho = floor(p/I) mod cp, local index l (see cp_kv_interleave_layout), i.e. to
 * k_cache[rho][block_tables[rho][b][l/block_size]][h][l mod block_size][:] (same for v).
 *   cu_new, start_pos  device int32 [B+1], [B];  block_tables device int32 [cp][B][max_blocks].
 *   k_cache, v_cache   device [cp][pool_pages][Hkv][block_size][d] of `dtype`.
 *   err  device int32 or NULL: CP_ERR_DEVICE_BOUNDS for a row whose table entry is missing
 *        or outside the pool (that row is not written).
 * A pure copy: bit-exact.  Rows of different calls that map to the same slot race.
 * ---------------------------------------------------------------------------- */
cp_status cp_kv_cache_write(const void* k_new, const void* v_new, const int32_t* cu_new,
                           const int32_t* start_pos, int32_t num_seqs, int32_t total_new,
                           int32_t num_kv_heads, int32_t head_dim, int32_t dtype, int32_t cp,
                           int32_t interleave, int32_t block_size, const int32_t* block_tables,
                           int32_t max_blocks, int64_t pool_pages, void* k_cache, void* v_cache,
                           int32_t* err, void* stream);

/* ------------------------------------------------------------------------------
 * cp_select_prefill_mode -- pass-KV or pass-Q for a prefill chunk ([PKV] Purpose: passing KV
 * suits full prefill because a KV head serves more than two query heads in most models; passing
 * Q suits chunked prefill when the cached context is much longer than the new queries).
 *
 * The pages' rule weighs the bytes ranks exchange; on one GPU nothing is exchanged and the
 * choice is the faster kernel for the shape.  The answer comes from a table measured on one
 * GB300 (partials + merge step of each mode, cp = 4, d = 128, bf16) over q_len in
 * {256, 1024, 4096}, kv_len / q_len in {1, 2, 4, 8, 16, 32} and q heads per kv head G in
 * {1, 2, 4, 8}; a shape takes its nearest grid point (log2 scale).  The two modes were within
 * 5% of each other almost everywhere: CP_PASS_Q is returned only where it was more than 3%
 * faster (q_len ~ 256 with kv_len ~ 2 q_len; G = 1 with q_len ~ 4096 and kv_len <= ~8 q_len),
 * CP_PASS_KV elsewhere.  Both modes run for every shape the library accepts (PASS_KV takes a
 * cached context through cu_seqlens_kv); which kv layout the caller holds decides which call
 * applies.  Host-only and pure; kv_len counts cached + new tokens, q_len the new ones;
 * head_dim and elem_bytes are accepted for the signature and do not change the answer.
 * ---------------------------------------------------------------------------- */
int32_t cp_select_prefill_mode(int64_t q_len, int64_t kv_len, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t elem_bytes);

/* ------------------------------------------------------------------------------
 * cp_partial_attn_prefill -- partial attention for every (Q shard, KV shard) pair
 * ([PKV] Purpose: pass-KV for full prefill, pass-Q for chunked prefill; the
 * exchange itself is logical here, so one launch covers every rotation step).
 *
 * PASS_KV (full prefill, or chunked prefill over a contiguous cached context):
 *   sequence b has q_len_b = cu_seqlens_q[b+1]-cu_seqlens_q[b] new queries and
 *   kv_len_b = cu_seqlens_kv[b+1]-cu_seqlens_kv[b] kv tokens (cached + new; NULL
 *   cu_seqlens_kv means kv_len_b = q_len_b, plain self-attention), token-major in k / v;
 *   query i sits at position C_b + i, C_b = kv_len_b - q_len_b (a sequence with
 *   C_b < 0 is flagged CP_ERR_DEVICE_BOUNDS in err and skipped).  The kv tokens are cut
 *   into 2cp chunks like cp_partition does (bounds floor(k*kv_len_b/(2cp))) and kv
 *   shard s = kv chunks s and 2cp-1-s.  Partial s of a query is its attention over the
 *   keys of kv shard s with position <= its own.  Q rows of shard r are chunks r and
 *   2cp-1-r of the new queries.
 * PASS_Q (chunked prefill over a paged, round-robin cache):
 *   sequence b has q_len_b = cu_seqlens_q[b+1]-cu_seqlens_q[b] new queries at
 *   positions C_b .. C_b+q_len_b-1, C_b = seq_lens_kv[b] - q_len_b, and
 *   seq_lens_kv[b] kv tokens (cached + new, already written) placed as in
 *   cp_kv_interleave_layout.  Partial r of a query is its attention over rank r's
 *   resident tokens with position <= its own.  Q rows of shard r are chunks r and
 *   2cp-1-r of the new tokens (the math does not depend on this split).
 *
 * Outputs: out[p][row][h][:] f32 (normalised over partial p's keys) and
 * lse[p][row][h] f32, p = kv shard / kv rank, row = token-major query row.  A
 * (row, partial) with no visible key gets lse = -inf and its out row holds zeros or
 * is left unwritten (the merge never reads it).
 * q_shard / kv_shard >= 0 restrict the launch to that Q shard / KV shard (one
 * logical rotation step); outputs of other pairs are left untouched.
 * ---------------------------------------------------------------------------- */
typedef struct cp_prefill_args {
  int32_t mode;                 /* cp_mode                                              */
  int32_t dtype;                /* cp_dtype of q, k, v, k_cache, v_cache                */
  int32_t impl;                 /* cp_impl                                              */
  int32_t num_seqs;             /* B >= 1                                               */
  int32_t num_q_heads;          /* Hq, multiple of num_kv_heads                         */
  int32_t num_kv_heads;         /* Hkv                                                  */
  int32_t head_dim;             /* d in {64, 128}                                       */
  int32_t cp;                   /* logical ranks, 1..64                                 */
  int32_t max_seqlen_q;         /* host: max new-query tokens of a sequence            */
  float softmax_scale;          /* <= 0 selects 1/sqrt(head_dim)                        */
  const int32_t* cu_seqlens_q;  /* device [B+1] token-major query rows                  */
  const int32_t* seq_lens_kv;   /* PASS_Q: device [B] cached + new kv tokens            */
  const void* q;                /* device [Nq][Hq][d]                                   */
  const void* k;                /* PASS_KV: device [Nkv][Hkv][d] (Nkv = total_kv or Nq) */
  const void* v;                /* PASS_KV: device [Nkv][Hkv][d]                        */
  const void* k_cache;          /* PASS_Q: device [cp][pool_pages][Hkv][block_size][d]  */
  const void* v_cache;          /* PASS_Q: same layout as k_cache                       */
  int64_t pool_pages;           /* PASS_Q: pages in each rank's pool                    */
  const int32_t* block_tables;  /* PASS_Q: device [cp][B][max_blocks] page ids          */
  int32_t max_blocks;           /* PASS_Q                                               */
  int32_t block_size;           /* PASS_Q: 16                                           */
  int32_t interleave;           /* PASS_Q: I >= 1                                       */
  int32_t q_shard;              /* -1 = all                                             */
  int32_t kv_shard;             /* -1 = all                                             */
  int32_t total_q;              /* host: Nq = cu_seqlens_q[B], rows of q/out/lse        */
  int32_t debug;                /* 0.  Testing only (tcgen05 kernel): 1 withholds the V */
                                /* tiles and shortens the wait budget so the pipeline's */
                                /* bounded waits expire -> CP_ERR_TIMEOUT in err        */
  float* out;                   /* device [cp][Nq][Hq][d] f32                           */
  float* lse;                   /* device [cp][Nq][Hq] f32                              */
  int32_t* err;                 /* device int32 or NULL                                 */
  const int32_t* cu_seqlens_kv; /* PASS_KV: device [B+1] kv rows of k / v, or NULL      */
  int32_t total_kv;             /* PASS_KV with cu_seqlens_kv: host, rows of k / v      */
  int32_t reserved;             /* 0                                                    */
} cp_prefill_args;

cp_status cp_partial_attn_prefill(const cp_prefill_args* args, void* stream);

/* ------------------------------------------------------------------------------
 * cp_attn_prefill_fused -- prefill with the merge folded in ([PKV] Purpose: the partials of
 * all KV shards / ranks of a Q row are combined; here one work item walks every shard's keys
 * with one online softmax, so no partial is written).  CP_PASS_KV: for a query tile of chunk c
 * the union of the shards' visible keys is the contiguous range of earlier positions.
 * CP_PASS_Q: the item walks the resident pages of rank 0, 1, .., cp-1 in turn through their
 * block tables ([PCP] Purpose), each row seeing a rank's tokens up to its own position.
 *
 * Same arguments as cp_partial_attn_prefill with dtype CP_BF16 and q_shard = kv_shard = -1
 * (args->out / args->lse are not used; CP_PASS_Q with impl CP_IMPL_TCGEN05_SINGLE is
 * CP_ERR_UNSUPPORTED); writes
 *   out      device bf16 [Nq][Hq][d]: exact causal attention (round to nearest even)
 *   out_lse  device f32 [Nq][Hq] natural-log LSE (NULL not allowed).
 * Equals cp_lse_merge applied to cp_partial_attn_prefill's partials, up to rounding.
 *
 * Tail split (CP_PASS_Q): its work items cost about the same, so when the grid's last wave
 * would leave SMs idle, the items of that wave are each cut into k rank ranges (rank
 * subsets of the walk) whose normalised partials and LSEs go to `workspace`; a second,
 * small kernel merges them as cp_lse_merge does.  cp_prefill_fused_workspace_size gives the
 * bytes this takes for the shapes in args on the current device (0: no split planned).
 * workspace: device scratch, 256-byte aligned, of at least that size; NULL, or a smaller
 * size, runs every item whole (same results up to rounding).  No initialisation is needed;
 * calls that use the same workspace must not overlap on the GPU.  CP_PASS_KV never splits.
 * ---------------------------------------------------------------------------- */
cp_status cp_prefill_fused_workspace_size(const cp_prefill_args* args, size_t* bytes);
cp_status cp_attn_prefill_fused(const cp_prefill_args* args, void* workspace,
                                size_t workspace_bytes, void* out, float* out_lse, void* stream);

/* ------------------------------------------------------------------------------
 * cp_partial_attn_decode -- per-rank partial attention of one new query token per
 * sequence over a round-robin paged cache ([PKV] Purpose: allgather decode, KV
 * round-robin on the ranks; [PCP] Purpose: per-rank block tables).
 *
 * The query of sequence b is at position seq_lens[b]-1 (its own kv entry is
 * already cached) and attends every token of the sequence; rank r's share is its
 * L_r resident tokens (local indices 0..L_r-1, see cp_kv_interleave_layout), cut
 * into num_splits ranges of split_tokens local tokens.  Partial p = r*num_splits+s.
 *
 *   q       device [B][Hq][d];  k_cache/v_cache as in cp_prefill_args.
 *   out     device f32 [cp*num_splits][B][Hq][d]; lse f32 [cp*num_splits][B][Hq].
 * Every split range must be covered: num_splits*split_tokens >= max_r L_r, which
 * cp_decode_plan guarantees; split_tokens is a multiple of block_size.
 * ---------------------------------------------------------------------------- */
typedef struct cp_decode_args {
  int32_t dtype;                /* cp_dtype of q and caches                             */
  int32_t num_seqs;             /* B                                                    */
  int32_t num_q_heads;          /* Hq = G * Hkv, G in 1 .. 16 (bf16) or 1 .. 8 (f32)    */
  int32_t num_kv_heads;         /* Hkv                                                  */
  int32_t head_dim;             /* d in {64, 128}                                       */
  int32_t cp;                   /* logical ranks                                        */
  int32_t interleave;           /* I                                                    */
  int32_t block_size;           /* 16                                                   */
  int32_t num_splits;           /* >= 1                                                 */
  int32_t split_tokens;         /* rank-local tokens per split                          */
  float softmax_scale;          /* <= 0 selects 1/sqrt(head_dim)                        */
  int32_t max_blocks;           /* columns of block_tables                              */
  int64_t pool_pages;           /* pages in each rank's pool                            */
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;  /* device [cp][B][max_blocks]                           */
  const int32_t* seq_lens;      /* device [B], 1 <= seq_lens[b] <= max_seq_len          */
  float* out;
  float* lse;
  int32_t* err;
} cp_decode_args;

/* Host-side split planning: picks split_tokens (multiple of block_size) and
 * num_splits so that num_splits*split_tokens covers the largest rank share of a
 * sequence of max_seq_len tokens and the grid fills the GPU. */
cp_status cp_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t cp, int32_t interleave,
                         int32_t block_size, int32_t max_seq_len, int32_t* num_splits,
                         int32_t* split_tokens);

cp_status cp_partial_attn_decode(const cp_decode_args* args, void* stream);

/* ------------------------------------------------------------------------------
 * cp_decode_attention -- decode partial attention and its LSE merge in one launch
 * ([PKV] Purpose: allgather decode -- every rank's partial, then their combination).
 *
 * Same inputs as cp_partial_attn_decode (args->out and args->lse are not used).  The
 * cp * num_splits partials go to `workspace`; the last CTA to finish for a (sequence, kv
 * head) merges them (as cp_lse_merge) and writes
 *   out      device [B][Hq][d], dtype of q (bf16: round to nearest even)
 *   out_lse  device f32 [B][Hq] or NULL.
 * Requires cp * num_splits <= 256.
 * workspace: device scratch of at least cp_decode_workspace_size() bytes, 256-byte aligned,
 * zero-filled before its first use (the call leaves it reusable: its counters return to
 * zero).  Calls that use the same workspace must not overlap on the GPU.
 * ---------------------------------------------------------------------------- */
cp_status cp_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t cp, int32_t num_splits,
                                   size_t* bytes);
cp_status cp_decode_attention(const cp_decode_args* args, void* workspace, size_t workspace_bytes,
                              void* out, float* out_lse, void* stream);

/* ------------------------------------------------------------------------------
 * cp_lse_merge -- combine P partials into exact attention (the combine step after
 * partial attention, [PKV] Purpose).
 *
 *   M = max_p lse_p;  w_p = exp(lse_p - M) (0 for lse_p = -inf);
 *   out = sum_p w_p * out_p / sum_p w_p;  out_lse = M + log(sum_p w_p).
 * A partial with lse = -inf contributes nothing: its out rows may hold anything (they
 * are never used; with few partials they may still be loaded).  All partials empty gives
 * out = 0 and out_lse = -inf.
 *
 *   partial_out  device f32 [P][rows][H][d];  partial_lse device f32 [P][rows][H].
 *   out          device [rows][H][d] of out_dtype (bf16: round to nearest even).
 *   out_lse      device f32 [rows][H] or NULL.
 * Stream-ordered like every call; the kernel is launched as a programmatic dependent of the
 * kernel before it on the stream (its blocks may be scheduled while that kernel finishes and
 * wait for its completion before reading anything).
 * ---------------------------------------------------------------------------- */
cp_status cp_lse_merge(const float* partial_out, const float* partial_lse, int32_t num_partials,
                       int64_t rows, int32_t num_heads, int32_t head_dim, void* out,
                       int32_t out_dtype, float* out_lse, void* stream);

/* ------------------------------------------------------------------------------
 * cp_decode_attention_noalloc -- cp_decode_attention for callers that cannot allocate
 * device memory when they call (no counterpart on the pages: it exists for this library's
 * users).
 *
 * Some callers have no device memory to give: a host framework that owns the whole GPU
 * memory pool and hands out none after start-up, or a fixed-footprint serving process that
 * must not allocate per request.  This entry point takes the same arguments as
 * cp_decode_attention minus the workspace and uses instead a scratch array built into the
 * library (CP_NOALLOC_SCRATCH_BYTES = 48 MiB per GPU).  The array lives in a module of its own:
 * a process holds it on a GPU from its first call of this entry point there until it exits;
 * the other entry points never load it.  It allocates and frees nothing.
 *   - Sizes whose scratch (cp_decode_workspace_size) exceeds CP_NOALLOC_SCRATCH_BYTES are
 *     rejected with CP_ERR_INVALID_ARG and a message naming both sizes.
 *   - The first call in a CUDA context looks up the array's device address (with that
 *     context's device current) and loads the array's module; make that first call before
 *     any stream capture.  A context that is destroyed and recreated (cudaDeviceReset) is
 *     recognised by its context id, and its first call looks the address up again.
 *   - Every call shares the one array: calls that overlap on the GPU (other streams, other
 *     threads) race and must be serialised by the caller.  Each call clears the array's
 *     arrival counters on `stream` before its launch.
 * ---------------------------------------------------------------------------- */
#define CP_NOALLOC_SCRATCH_BYTES (48u * 1024u * 1024u)
cp_status cp_decode_attention_noalloc(const cp_decode_args* args, void* out, float* out_lse,
                                      void* stream);

/* sizeof() of the argument structs, so bindings can check their mirror. */
size_t cp_prefill_args_size(void);
size_t cp_decode_args_size(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
