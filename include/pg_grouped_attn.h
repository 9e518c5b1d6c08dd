/*
 * Grouped attention over packed shared-prefix sequences (Prefix Grouper), forward and backward,
 * for NVIDIA GB300 (sm_103a).  Plain C ABI: host scalars, host or device pointers, sizes.
 *
 * What is computed.  A batch holds B groups.  Group b is packed as [P_b; R_b1; ...; R_bG]: a shared
 * prefix of Lp_b tokens followed by its G_b responses back to back ("Sequential Concatenation",
 * skill page "prefix-grouper-grpo", Architecture Overview; Pith review of Prefix Grouper, "Core
 * claim").  Self-attention over that sequence is the grouped attention of the Pith review ("What
 * carries the argument"): prefix queries attend causally to the prefix only; a query of response i
 * attends to the whole prefix and causally to response i, never to another response; position IDs
 * are those of the repeated-prefix baseline, so every response restarts at Lp_b.  The result equals
 * running every [P_b; R_bi] through causal attention separately (abstract page: identical forward
 * outputs and backward gradients), with the shared prefix computed once, and in the backward the
 * prefix K/V gradient summed over all responses of the group.
 *
 * Tensor layout (all row-major, head_dim contiguous, packed token order, T = total tokens):
 *   q, o, dO, dq   [T, Hq,  d]
 *   k, v, dk, dv   [T, Hkv, d]      query head h uses key/value head h / (Hq / Hkv)
 *   lse            [Hq, T]  fp32, natural-log log-sum-exp of each query row's scaled scores
 * Element type: PG_F32 (fp32 in, fp32 out, fp32 arithmetic) or PG_BF16 (bf16 in and out, fp32
 * accumulation; rotated Q/K and softmax probabilities are rounded to bf16 before the tensor-core
 * products).
 *
 * Ownership.  The caller allocates and owns every buffer (inputs, outputs, the packed-layout tables,
 * the workspace) and every stream.  The library allocates no device memory and keeps no host state
 * other than a per-thread error message and one device status word.
 *
 * Execution.  Every call that takes a stream is asynchronous on it; argument checks happen on the
 * host before any launch and return an error without launching anything.  Errors found by kernels
 * (a bounded wait that ran out) are recorded in the device status word; read it with
 * pg_device_status after synchronising.
 */
#ifndef PG_GROUPED_ATTN_H
#define PG_GROUPED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pg_stream_t; /* the same type as cudaStream_t; NULL = legacy stream */

typedef enum pg_status {
  PG_OK = 0,
  PG_ERR_INVALID_ARG = 1,   /* bad length, head count, head_dim, alignment, pointer or size */
  PG_ERR_UNSUPPORTED = 2,   /* a valid request with no kernel (never silently emulated) */
  PG_ERR_CUDA = 3,          /* a CUDA runtime call failed; see pg_last_error_message */
  PG_ERR_TIMEOUT = 4,       /* a kernel's bounded wait ran out (reported by pg_device_status) */
  PG_ERR_DEVICE = 5         /* a kernel-side check failed (reported by pg_device_status) */
} pg_status;

typedef enum pg_dtype { PG_F32 = 0, PG_BF16 = 1 } pg_dtype;

/* Options for the attention calls.  A zeroed struct (or NULL) means: scale d^-1/2, no RoPE. */
typedef struct pg_opts {
  float softmax_scale;  /* 0 => head_dim^-1/2 (the skill page's sketch divides by sqrt(head_dim)) */
  float rope_theta;     /* 0 => no RoPE; else rotate-half RoPE, angle pos * theta^(-2k/d) */
  uint32_t flags;       /* PG_FLAG_* below */
  uint32_t debug;       /* 0 in normal use; PG_DEBUG_* below */
} pg_opts;

/* Run the fp32-arithmetic SIMT kernels even for bf16 inputs (a slower, independent path). */
#define PG_FLAG_SIMT 1u

/*
 * Forward only: compute o and lse for the response rows alone, for scoring many short responses
 * against one long shared context (Pith review, "Core claim": judging many short questions against
 * one long context reuses the same sharing pattern).  Every response row still attends to its whole
 * prefix and causally to its own response, so k and v must hold the prefix rows too (for example a
 * cached context); the prefix rows of o and lse are not written and their q rows are not read.
 * Rejected by pg_grouped_attn_bwd (PG_ERR_INVALID_ARG).  The bf16, head_dim 128 kernel packs the
 * Hq / Hkv query heads that share a key/value head into one tile and splits the prefix keys across
 * CTAs, so each prefix K/V row is read from memory about once per key/value head; the partial
 * results are merged by their log-sum-exp in a second kernel (workspace: pg_workspace_size with
 * this flag).
 */
#define PG_FLAG_RESPONSES_ONLY 2u

/*
 * Backward with dq bitwise reproducible as well: the bf16 head_dim-128 path computes dq in a
 * query-major tensor-core kernel (each row's dq summed by one CTA in a fixed key order, then
 * inverse-rotated and cast in its epilogue) and dk / dv in the key-major kernel without its dQ
 * part.  Without the flag dq is accumulated across key blocks with TMA reduce-adds (fp32, summation
 * order not fixed).  The fp32 / SIMT path is deterministic either way.
 */
#define PG_FLAG_DETERMINISTIC 4u

/*
 * Rotate q and k once per training step instead of twice: with this flag pg_grouped_attn_fwd writes
 * the RoPE-rotated q and k and the cos/sin table into its workspace, laid out as the backward's
 * workspace (so it must be at least pg_workspace_size(..., phase 1) bytes), and
 * pg_grouped_attn_bwd with the flag reads them from there instead of rotating again.  On the bf16
 * tensor-core path the forward also leaves the backward its log2-domain LSE rows.  Pass the
 * backward the same
 * workspace, unmodified since the forward, with the same layout, q, k, heads, rope_theta and flags.
 * Without RoPE the flag changes nothing.
 */
#define PG_FLAG_KEEP_ROTATED 8u

/*
 * q and k arrive already RoPE-rotated at the layout's position ids with opts->rope_theta (for
 * example by pg_gemm_bf16_rope in the projection that produced them, from the table pg_rope_table
 * wrote): the calls do not rotate them again.  The backward still returns dq and dk with respect
 * to the un-rotated q and k (rotating them back with the cos/sin table), exactly as without the
 * flag, so the table must be in the workspace: call pg_rope_table on the backward's workspace
 * (same layout, heads, rope_theta and flags) before the forward, and keep it unchanged until the
 * backward.  Needs rope_theta > 0 (PG_ERR_INVALID_ARG otherwise).  Combines with
 * PG_FLAG_KEEP_ROTATED (the forward then leaves only its LSE rows for the backward),
 * PG_FLAG_DETERMINISTIC, PG_FLAG_SIMT and PG_FLAG_RESPONSES_ONLY.
 */
#define PG_FLAG_PRE_ROTATED 16u

/* Test hook for the bounded-wait error path: the tensor-core forward never signals that P is
 * ready, so its MMA thread's wait runs out (after 50 ms instead of 2 s), the kernel records
 * PG_ERR_TIMEOUT in the status word and exits cleanly; the outputs are then undefined. */
#define PG_DEBUG_WITHHOLD_P 1u

/*
 * Host-side summary of a packed batch, filled by pg_pack / pg_pack_host.  The two pointers refer to
 * the caller's buffers (device buffers for pg_pack, host buffers for pg_pack_host) which must stay
 * alive and unchanged while the layout is used.  All other fields are informational or sizes.
 */
typedef struct pg_layout {
  int64_t num_groups;      /* B */
  int64_t num_segments;    /* total responses, sum of G_b */
  int64_t total_tokens;    /* T */
  int64_t max_position;    /* 1 + the largest position id */
  int64_t pairs;           /* visible (query, key) pairs per head, summed over groups */
  int64_t n_tiles[6];      /* work-list lengths: fwd 64-row, fwd 128-row, bwd 64-key, bwd 128-key,
                              fwd 256-row, response spans (one per group with response rows) */
  int64_t off_tiles[6];    /* byte offsets of those lists in the tables */
  int64_t off_tokens;      /* byte offset of the per-token table (16 bytes per token) */
  int64_t table_bytes;     /* bytes of the tables buffer in use */
  const int32_t* position_ids; /* [T] */
  const void* tables;
  int64_t max_response_rows; /* the largest number of response rows (sum of R_bi) in one group */
  int64_t n_pad_rows;      /* padded layouts (pg_pack_padded): number of padding rows, else 0 */
  int64_t off_pad_rows;    /* byte offset of the padding rows' indices (int32) in the tables */
  int64_t max_depth;       /* segments on the longest root-to-leaf path: 1 (prefixes only) or 2
                              for pg_pack layouts, up to 8 for pg_pack_tree layouts */
  int64_t n_intervals;     /* entries (2 x int32 key ranges) of the tiles' interval table */
  int64_t off_intervals;   /* its byte offset in the tables */
} pg_layout;

/*
 * Sizes needed for a packed batch.  prefix_lens[num_groups], group_sizes[num_groups] and
 * suffix_lens[sum(group_sizes)] are host arrays (responses listed group by group).  Returns
 * T = Lp_0 + sum(R_0i) + ... in *total_tokens and the bytes the tables need in *table_bytes.
 * Errors: PG_ERR_INVALID_ARG if num_groups < 1, any length or group size < 0, T == 0 or T >= 2^30.
 */
pg_status pg_pack_size(int32_t num_groups, const int32_t* prefix_lens, const int32_t* group_sizes,
                       const int32_t* suffix_lens, int64_t* total_tokens, int64_t* table_bytes);

/*
 * Build the packed layout on the host (no CUDA call): position_ids[T] (prefix token j -> j,
 * token j of a response -> Lp + j, as in the repeated-prefix baseline: Pith review, "What carries
 * the argument"), the per-token visibility table and the tile work-lists, into caller host buffers
 * position_ids (int32 [T]) and tables (table_bytes >= pg_pack_size's), and fill *layout.
 * Per-token table entry t (4 x int32): {g0, pe, own_lo, pos}: the group's first row, the row after
 * its prefix, the first row of the token's own response (g0 for prefix tokens) and its position.
 * Query row t sees key row s iff  s <= t && s >= g0 && (s < pe || s >= own_lo).
 * Errors: as pg_pack_size, plus PG_ERR_INVALID_ARG for NULL buffers or a short table buffer.
 */
pg_status pg_pack_host(int32_t num_groups, const int32_t* prefix_lens, const int32_t* group_sizes,
                       const int32_t* suffix_lens, int32_t* position_ids, void* tables,
                       int64_t table_bytes, pg_layout* layout);

/*
 * pg_pack_host into a temporary host buffer, then asynchronous copies to the caller's device
 * buffers position_ids_dev (int32 [T]) and tables_dev (table_bytes) on `stream`; *layout points at
 * the device buffers.  The host staging is released before return (pageable copies are staged
 * synchronously by CUDA), so the call is safe to follow by kernels on the same stream.
 * Errors: as pg_pack_host; PG_ERR_CUDA if a copy fails.
 */
pg_status pg_pack(int32_t num_groups, const int32_t* prefix_lens, const int32_t* group_sizes,
                  const int32_t* suffix_lens, int32_t* position_ids_dev, void* tables_dev,
                  int64_t table_bytes, pg_layout* layout, pg_stream_t stream);

/*
 * Nested prefixes (Pith review, "Reading between the lines": multi-turn histories shared by many
 * continuations).  num_nodes segments with seg_lens[i] tokens each; parent[i] is the index of
 * segment i's parent (-1 for a root), and the segments are listed in depth-first preorder (a parent
 * before its children, a subtree contiguous), which is also their packed row order.  A token sees
 * every token of its segment's ancestors and the tokens of its own segment up to itself; its
 * position id is the total length of its ancestors plus its offset in its segment -- its position
 * in the root-to-leaf sequence the repeated-prefix baseline would run.  Each root is a group; a root
 * whose children are all leaves is exactly a pg_pack group.  The attention calls then compute that
 * attention, and in the backward every segment's gradient sums over all continuations below it.
 * Buffers and errors as pg_pack_size / pg_pack_host / pg_pack; PG_ERR_INVALID_ARG for a negative
 * length or an order that is not a depth-first preorder, PG_ERR_UNSUPPORTED for a nesting depth
 * (segments on a root-to-leaf path) above 8.  PG_FLAG_RESPONSES_ONLY needs depth <= 2.
 */
pg_status pg_pack_tree_size(int32_t num_nodes, const int32_t* parent, const int32_t* seg_lens,
                            int64_t* total_tokens, int64_t* table_bytes);
pg_status pg_pack_tree_host(int32_t num_nodes, const int32_t* parent, const int32_t* seg_lens,
                            int32_t* position_ids, void* tables, int64_t table_bytes,
                            pg_layout* layout);
pg_status pg_pack_tree(int32_t num_nodes, const int32_t* parent, const int32_t* seg_lens,
                       int32_t* position_ids_dev, void* tables_dev, int64_t table_bytes,
                       pg_layout* layout, pg_stream_t stream);

/*
 * Padded layout (skill page "prefix-grouper-grpo", Step 3 "Restructure Input Format"): each of the
 * num_groups groups is [P; slot_1; ...; slot_G] with prefix_len prefix tokens and group_size slots
 * of max_response_len tokens; response i of group b fills the first response_lens[b * group_size +
 * i] tokens of its slot and the rest of the slot is padding (where that page's attention mask is 0).
 * Padding only ever trails a response, so causal attention never lets a real token see it: the
 * padded buffer is run as a packed layout whose responses all have max_response_len tokens (so
 * positions, tiles and pairs count the padding too), and the layout also lists the padding rows.
 * With such a layout pg_grouped_attn_fwd writes o = 0 and lse = +inf on padding rows (+inf makes
 * exp(s - lse) = 0, so in the backward a padding query has no weight: its dO must be finite but
 * is otherwise ignored) and pg_grouped_attn_bwd writes dq = dk = dv = 0 on them.  Real rows get the
 * results of the unpadded packing.  Padding rows still cost kernel time in proportion to their
 * number.  Buffers and errors as pg_pack_size / pg_pack_host / pg_pack; additionally
 * PG_ERR_INVALID_ARG if a response length is outside [0, max_response_len].
 */
pg_status pg_pack_padded_size(int32_t num_groups, int32_t prefix_len, int32_t group_size,
                              int32_t max_response_len, const int32_t* response_lens,
                              int64_t* total_tokens, int64_t* table_bytes);
pg_status pg_pack_padded_host(int32_t num_groups, int32_t prefix_len, int32_t group_size,
                              int32_t max_response_len, const int32_t* response_lens,
                              int32_t* position_ids, void* tables, int64_t table_bytes,
                              pg_layout* layout);
pg_status pg_pack_padded(int32_t num_groups, int32_t prefix_len, int32_t group_size,
                         int32_t max_response_len, const int32_t* response_lens,
                         int32_t* position_ids_dev, void* tables_dev, int64_t table_bytes,
                         pg_layout* layout, pg_stream_t stream);

/*
 * Workspace bytes for pg_grouped_attn_fwd (phase 0) or pg_grouped_attn_bwd (phase 1) with this
 * layout, dtype, head counts, head_dim and options.  Deterministic in its arguments.
 */
pg_status pg_workspace_size(const pg_layout* layout, pg_dtype dtype, int32_t heads_q,
                            int32_t heads_kv, int32_t head_dim, const pg_opts* opts, int32_t phase,
                            size_t* bytes);

/*
 * Grouped attention forward (the prefix self-attention and the suffix attention of the Pith
 * review's two-call decomposition, "What carries the argument", computed in one pass over the
 * packed layout).  Inputs q [T,Hq,d], k, v [T,Hkv,d] (device); outputs o [T,Hq,d] and
 * lse [Hq,T] fp32 (device), every element written.  workspace: device, >= pg_workspace_size(...,0).
 * RoPE, when enabled, rotates q and k by the layout's position ids before the products; o is not
 * rotated.  Requirements: Hq % Hkv == 0, d in {64, 128}, 16-byte aligned pointers.
 * Errors: PG_ERR_INVALID_ARG (checked on the host, nothing launched); PG_ERR_UNSUPPORTED for a
 * dtype / head_dim with no kernel; PG_ERR_CUDA if a launch fails.
 */
pg_status pg_grouped_attn_fwd(const pg_layout* layout, pg_dtype dtype, int32_t heads_q,
                              int32_t heads_kv, int32_t head_dim, const void* q, const void* k,
                              const void* v, void* o, float* lse, const pg_opts* opts,
                              void* workspace, size_t workspace_bytes, pg_stream_t stream);

/*
 * Grouped attention backward for the loss sum(dO * o): gradients dq [T,Hq,d], dk, dv [T,Hkv,d]
 * (device, every element written, dtype of the inputs) with respect to the un-rotated q, k and v.
 * A prefix key's dk/dv sums the contributions of the prefix queries and of every response of its
 * group (Pith review, Appendix A.1 objection: the single shared prefix's gradient equals the sum
 * over the G baseline copies), in a fixed order, so dk and dv are bitwise reproducible.
 * o and lse are the forward's outputs for the same inputs and options.
 * Errors: as pg_grouped_attn_fwd, with workspace >= pg_workspace_size(..., 1).
 */
pg_status pg_grouped_attn_bwd(const pg_layout* layout, pg_dtype dtype, int32_t heads_q,
                              int32_t heads_kv, int32_t head_dim, const void* q, const void* k,
                              const void* v, const void* o, const float* lse, const void* dO,
                              void* dq, void* dk, void* dv, const pg_opts* opts, void* workspace,
                              size_t workspace_bytes, pg_stream_t stream);

/*
 * RoPE cos/sin table for PG_FLAG_PRE_ROTATED: writes (cos a, sin a), a = position_ids[t] *
 * rope_theta^(-2k/d), as float2 [T][d/2] (row t, column k; fp32) into `workspace` -- the
 * workspace later passed to pg_grouped_attn_bwd (and, with PG_FLAG_KEEP_ROTATED, to
 * pg_grouped_attn_fwd) with the same layout, dtype, heads and opts, where the table occupies the
 * first T * d/2 * 8 bytes -- and returns its device address in *table (for pg_gemm_bf16_rope).
 * opts must carry rope_theta > 0 and PG_FLAG_PRE_ROTATED; workspace >= pg_workspace_size(..., 1),
 * 16-byte aligned.  Asynchronous on `stream`.
 * Errors: PG_ERR_INVALID_ARG (host check, nothing launched); PG_ERR_CUDA on a launch failure.
 */
pg_status pg_rope_table(const pg_layout* layout, pg_dtype dtype, int32_t heads_q, int32_t heads_kv,
                        int32_t head_dim, const pg_opts* opts, void* workspace,
                        size_t workspace_bytes, const void** table, pg_stream_t stream);

/* Kernels of the library, for pg_set_profile. */
typedef enum pg_kernel {
  PG_KERNEL_NONE = 0,
  PG_KERNEL_ROPE = 1,            /* RoPE of q and k (forward rotation) */
  PG_KERNEL_ATTN_FWD = 2,        /* the grouped-attention forward */
  PG_KERNEL_BWD_PREPROCESS = 3,  /* rowsum(dO * O) */
  PG_KERNEL_BWD_DKDV = 4,        /* key-major dK/dV (and dQ where fused) */
  PG_KERNEL_BWD_DQ = 5,          /* query-major dQ */
  PG_KERNEL_ROPE_BWD = 6,        /* inverse RoPE of dQ/dK and the cast to the output dtype */
  PG_KERNEL_GEMM = 7,            /* the bf16 tensor-core GEMM (decoder-layer path) */
  PG_KERNEL_LAYER = 8,           /* RMSNorm / SwiGLU kernels of the decoder-layer path */
  PG_KERNEL_SCORE_COMBINE = 9,   /* merge of the responses-only forward's key splits */
  PG_KERNEL_PAD_FILL = 10        /* padded layouts: outputs / gradients of the padding rows */
} pg_kernel;

/*
 * Profiling record.  While installed for a thread (pg_set_profile), every kernel launch the
 * library makes from that thread increments `launches`, and each launch of kernel `kernel` is
 * bracketed on the call's stream by cudaEventRecord(ev_begin) and cudaEventRecord(ev_end)
 * (cudaEvent_t handles owned by the caller; either may be NULL).  Measurement support only; it
 * changes nothing that is computed.
 */
typedef struct pg_profile {
  int32_t kernel;
  int32_t reserved;
  void* ev_begin;
  void* ev_end;
  int64_t launches;
} pg_profile;

/* Install (profile != NULL) or remove (NULL) the calling thread's profiling record.  The record
 * must outlive its installation. */
pg_status pg_set_profile(pg_profile* profile);

/* Size of the built-in scratch of pg_grouped_attn_fwd_noalloc: 16 MiB per GPU. */
#define PG_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * pg_grouped_attn_fwd without a workspace argument, for callers that cannot allocate device
 * memory: for example a host program that owns a fixed device-memory plan and hands this library
 * only the tensors it already holds, or code running at a point where a cudaMalloc would
 * synchronise the device or is not permitted.  The paper has no counterpart; this is a
 * deployment convenience.
 *
 * Scratch (the RoPE-rotated Q and K the kernel reads) comes from a 16 MiB array
 * (PG_NOALLOC_SCRATCH_BYTES) that the library reserves statically on every GPU it is loaded on,
 * for the life of the process.  A problem whose scratch would exceed it (pg_workspace_size(...,
 * phase 0) > PG_NOALLOC_SCRATCH_BYTES) is rejected with PG_ERR_INVALID_ARG before anything runs;
 * use pg_grouped_attn_fwd with a caller workspace for it.  Nothing here calls cudaMalloc,
 * cudaFree or any allocating routine.
 *
 * The first call on each device looks up the array's device address (with that device current)
 * and caches it; make that first call before any stream capture.  Every call shares the one array
 * and leaves its contents behind (no part of it needs to start at zero): calls that can overlap on
 * the GPU -- on different streams without ordering between them -- race on it and must not be
 * issued.  Arguments, results and errors are otherwise those of pg_grouped_attn_fwd.
 */
pg_status pg_grouped_attn_fwd_noalloc(const pg_layout* layout, pg_dtype dtype, int32_t heads_q,
                                      int32_t heads_kv, int32_t head_dim, const void* q,
                                      const void* k, const void* v, void* o, float* lse,
                                      const pg_opts* opts, pg_stream_t stream);

/*
 * Read (synchronously, on the current device) the status word kernels set when a bounded wait
 * runs out or a kernel-side check fails; PG_OK if none did.  clear != 0 resets it afterwards.
 */
pg_status pg_device_status(int32_t clear);

/* Static text for a status code. */
const char* pg_status_string(pg_status status);

/* The calling thread's last error message ("" if none). */
const char* pg_last_error_message(void);

#ifdef __cplusplus
}
#endif
#endif /* PG_GROUPED_ATTN_H */
