/*
 * lsx.h -- C ABI of liblsx: exact softmax attention computed blockwise over
 * sequence chunks, on one NVIDIA GB300 (sm_103a).
 *
 * The method (sources are the pages' titles and sections):
 *  - BurstAttention: An Efficient Distributed Attention Framework for
 *    Extremely Long Sequences -- method section: the sequence is split into
 *    chunks; each device computes "local attention" of its query chunk against
 *    key/value chunks and the local results are aggregated into global ones.
 *  - Lean Attention (abstract): the associative property of online softmax
 *    makes the combination of partial results a reduction.
 *  - Tree Attention: Topology-aware Decoding for Long-Context Attention on GPU
 *    clusters (abstract): the reduction across the sequence axis is computed
 *    as a tree reduction.
 *  - DistFlashAttn ("Effiziente verteilte Aufmerksamkeit ...", core concepts):
 *    load-balanced scheduling of causal work across workers, and a backward
 *    pass that reuses the saved attention output instead of re-running the
 *    forward pass.
 *
 * Conventions shared by every entry point
 *  - Tensors are rank-4 views [B, H, N, D] described by lsx_tensor.  The D
 *    axis is contiguous (stride 1); the other strides are in ELEMENTS.  A
 *    log-sum-exp tensor is an fp32 view with D == 1, 4-byte aligned, with
 *    any non-negative B/H/N strides (its stride along D is never used).
 *  - Every buffer is owned by the caller.  The library allocates no device or
 *    host memory; scratch space ("workspace") is passed in by the caller, who
 *    sizes it with the matching *_workspace_size call.  A workspace may be
 *    reused by the next call once that call's stream has reached it.
 *  - Pointers are DEVICE pointers unless an entry point says otherwise.
 *    Device data must be 16-byte aligned; for bf16 tensors fed to the tensor
 *    core path, every stride must also be a multiple of 8 elements.
 *  - Every call is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and returns without synchronising.
 *  - Return value: LSX_OK, or a negative LSX_ERR_* code.  A call that returns
 *    an error has launched nothing and touched no buffer.  A failure detected
 *    on the device (a bounded wait that ran out) is recorded in a per-device
 *    status word that lsx_sync_status reads back.
 *  - Softmax scale: scores are scale * <q_i, k_j>; scale <= 0 selects
 *    1/sqrt(D).  LSE is in natural-log units of the scaled scores.
 *  - Causal masking uses ABSOLUTE positions: query row i of a chunk that
 *    starts at q_off sees key row j of a chunk that starts at kv_off iff
 *    kv_off + j <= q_off + i.  A query with no visible key gets O = 0 and
 *    LSE = -inf, the identity of the merge.
 *  - Grouped query heads: query head h reads key/value head h / (Hq / Hkv).
 */
#ifndef LSX_H
#define LSX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* lsx_stream_t; /* identical to cudaStream_t */

enum lsx_dtype { LSX_BF16 = 0, LSX_F32 = 1 };

enum lsx_status {
  LSX_OK = 0,
  LSX_ERR_NULL = -1,        /* a required pointer is NULL                    */
  LSX_ERR_SHAPE = -2,       /* shapes disagree                               */
  LSX_ERR_DTYPE = -3,       /* dtype combination not supported               */
  LSX_ERR_ALIGN = -4,       /* base or stride alignment violated             */
  LSX_ERR_UNSUPPORTED = -5, /* valid request outside what is implemented     */
  LSX_ERR_WORKSPACE = -6,   /* workspace missing or too small                */
  LSX_ERR_LAUNCH = -7,      /* a CUDA launch or API call failed              */
  LSX_ERR_TIMEOUT = -8,     /* a device-side bounded wait ran out            */
  LSX_ERR_DEVICE = -9       /* no usable sm_103 device / context             */
};

typedef struct lsx_tensor {
  void* data;      /* base pointer (device unless stated otherwise)          */
  int32_t dtype;   /* enum lsx_dtype                                         */
  int32_t reserved;
  int64_t B, H, N, D;
  int64_t stride_b, stride_h, stride_n; /* elements; stride of D is 1        */
} lsx_tensor;

/* ------------------------------------------------------------------------
 * attn_chunk_fwd -- local attention of one (query chunk, key/value chunk)
 * pair (BurstAttention, method: local attention computation; Lean Attention,
 * abstract: online softmax).
 *   q  [B, Hq, Lq, D]    bf16 or f32
 *   k  [B, Hkv, Lk, D]   same dtype as q
 *   v  [B, Hkv, Lk, D]   same dtype as q
 *   o  [B, Hq, Lq, D]    out: bf16 or f32 (f32 inputs need f32 o)
 *   lse[B, Hq, Lq, 1]    out: f32, natural log
 * accumulate == 0: o, lse receive this pair's normalised partial.
 * accumulate == 1: o, lse hold a partial over other keys; the new partial is
 *   merged into them in the epilogue (the LSE-weighted merge of attn_merge).
 * D in {64, 128}.  bf16 inputs run on the tcgen05 tensor cores (fp32
 * accumulation, P rounded to bf16 for the P.V product); f32 inputs run an
 * fp32 CUDA-core path.
 * Workspace (bf16 only, optional): NULL, or at least
 * attn_chunk_fwd_workspace_size(q, k) bytes, 256-byte aligned.  With it, a
 * key-contiguous copy of V is written there first and the P.V product reads
 * that copy, which the tensor cores consume about twice as fast; without
 * it, V is read as stored.  Both give the same results.  A non-NULL
 * workspace that is too small returns LSX_ERR_WORKSPACE.
 * ---------------------------------------------------------------------- */
size_t attn_chunk_fwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k);
int attn_chunk_fwd(const lsx_tensor* q, const lsx_tensor* k,
                   const lsx_tensor* v, int64_t q_off, int64_t kv_off,
                   int causal, float scale, const lsx_tensor* o,
                   const lsx_tensor* lse, int accumulate, void* workspace,
                   size_t workspace_bytes, lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_merge -- LSE-weighted merge of two partials over disjoint key sets
 * (BurstAttention abstract: aggregate local results into global ones;
 * Lean Attention abstract: the merge is associative):
 *   LSE = m + log(exp(LSE_a - m) + exp(LSE_b - m)),  m = max(LSE_a, LSE_b)
 *   O   = exp(LSE_a - LSE) O_a + exp(LSE_b - LSE) O_b
 * o_a, o_b, o_out: [B, H, N, D] bf16 or f32 (each independently);
 * lse_*: [B, H, N, 1] f32.  o_out/lse_out may alias o_a/lse_a or o_b/lse_b
 * exactly (same base and strides).  Two -inf inputs give O = 0, LSE = -inf.
 * D in {64, 128}.
 * ---------------------------------------------------------------------- */
int attn_merge(const lsx_tensor* o_a, const lsx_tensor* lse_a,
               const lsx_tensor* o_b, const lsx_tensor* lse_b,
               const lsx_tensor* o_out, const lsx_tensor* lse_out,
               lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_tree_merge -- one-pass reduction of n_parts partials (Tree Attention
 * abstract: tree reduction across the sequence axis; DeFT abstract: global
 * reduction of partial attention).  Partial p of every row is combined in a
 * fixed order, so the result is bit-deterministic.
 *   o_parts:   [B, H, N, D] view of partial 0; partial p starts at
 *              data + p * part_stride_o elements (bf16 or f32)
 *   lse_parts: [B, H, N, 1] view of partial 0; partial p starts at
 *              data + p * part_stride_lse elements (f32)
 *   o_out [B, H, N, D] bf16 or f32; lse_out [B, H, N, 1] f32 (may be NULL
 *   data to skip writing LSE).
 * 1 <= n_parts <= 4096.  D in {64, 128}.
 * ---------------------------------------------------------------------- */
int attn_tree_merge(const lsx_tensor* o_parts, int64_t part_stride_o,
                    const lsx_tensor* lse_parts, int64_t part_stride_lse,
                    int n_parts, const lsx_tensor* o_out,
                    const lsx_tensor* lse_out, lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_chunk_bwd -- gradients of one chunk pair from the SAVED final output
 * and log-sum-exp, without re-running the forward pass (DistFlashAttn, core
 * concepts: rematerialization-aware gradient checkpointing).
 *   q, k, v as in attn_chunk_fwd; o [B,Hq,Lq,D] and lse [B,Hq,Lq,1] are the
 *   FINAL (fully merged) output and LSE of the query rows; d_o like o.
 *   dq [B,Hq,Lq,D], dk/dv [B,Hkv,Lk,D]: out, bf16 or f32.
 * accumulate == 0: outputs receive this pair's contribution.
 * accumulate == 1: the contribution is added to the outputs (use f32
 *   outputs to sum over many chunk pairs).
 * Workspace (256-byte aligned): at least attn_chunk_bwd_min_workspace_size
 * bytes (the row sums delta_i = <dO_i, O_i>, 4 bytes per query row).  With
 * attn_chunk_bwd_workspace_size bytes (bf16 inputs) more is kept there:
 * 16 bytes per query row of row statistics (-LSE/scale and -delta as bf16
 * triples), which the dK/dV products add to their score tiles on the tensor
 * cores instead of per element, and one scratch region used EITHER as the
 * fp32 dQ accumulator of the fused kernel (bf16 inputs; 4 bytes x B x Hq x Lq x
 * D; see lsx_set_deterministic) OR as a key-contiguous copy of K, which the
 * separate dQ kernel reads at the tensor cores' faster operand layout.
 * With less, the statistics are applied per element, K is read as stored,
 * and the fused kernel runs only when dq is f32 (it then adds into dq
 * directly).  All forms give results within the documented tolerance of
 * each other (the statistics triples carry 24 significant bits).
 * ---------------------------------------------------------------------- */
size_t attn_chunk_bwd_min_workspace_size(const lsx_tensor* q, const lsx_tensor* k);
size_t attn_chunk_bwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k);
int attn_chunk_bwd(const lsx_tensor* q, const lsx_tensor* k,
                   const lsx_tensor* v, const lsx_tensor* o,
                   const lsx_tensor* lse, const lsx_tensor* d_o,
                   int64_t q_off, int64_t kv_off, int causal, float scale,
                   const lsx_tensor* dq, const lsx_tensor* dk,
                   const lsx_tensor* dv, int accumulate, void* workspace,
                   size_t workspace_bytes, lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_block_sparse_fwd / attn_block_sparse_bwd -- exact attention over the
 * whole sequence restricted to a block mask (the Fine-grained Attention I/O
 * Complexity page, abstract: the analysis extends to sparse attention; the
 * BriefGPT BurstAttention page's related work: FlashAttention extended to a
 * broad class of sparsity patterns).  Tiles of masked blocks are skipped by
 * the same persistent kernels as attn_chunked_fwd / attn_chunked_bwd.
 *   block_mask: DEVICE pointer to uint8 [ceil(Lq/128)][ceil(Lk/128)],
 *     row-major, shared by every batch row and head; entry (i, j) nonzero
 *     lets query rows [128 i, 128 i + 128) see keys [128 j, 128 j + 128).
 *   causal: the causal rule (key position <= query position, both counted
 *     from 0) applies inside the allowed blocks as well.
 *   A query left with no visible key gets O = 0, LSE = -inf; in the
 *   backward its rows contribute nothing.
 *   q, k, v, o, d_o bf16 (LSX_ERR_DTYPE otherwise); dq, dk, dv bf16 or f32.
 *   Workspace (256-byte aligned, required): at least the matching
 *   *_workspace_size bytes (LSX_ERR_WORKSPACE otherwise).  The forward and
 *   backward are consistent with each other and with the chunked calls.
 * ---------------------------------------------------------------------- */
size_t attn_block_sparse_fwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k);
int attn_block_sparse_fwd(const lsx_tensor* q, const lsx_tensor* k, const lsx_tensor* v,
                          const uint8_t* block_mask, int causal, float scale,
                          const lsx_tensor* o, const lsx_tensor* lse, void* workspace,
                          size_t workspace_bytes, lsx_stream_t stream);
size_t attn_block_sparse_bwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k);
int attn_block_sparse_bwd(const lsx_tensor* q, const lsx_tensor* k, const lsx_tensor* v,
                          const lsx_tensor* o, const lsx_tensor* lse, const lsx_tensor* d_o,
                          const uint8_t* block_mask, int causal, float scale,
                          const lsx_tensor* dq, const lsx_tensor* dk, const lsx_tensor* dv,
                          void* workspace, size_t workspace_bytes, lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_chunk_bwd_noalloc -- attn_chunk_bwd for callers that cannot allocate
 * device memory when they call it (none of the cited methods has a
 * counterpart; this is a deployment convenience of the library).  Examples:
 * an extension running inside a host application that owns the device
 * memory pool and offers no way to request more, or a latency-critical loop
 * that forbids allocation after start-up.  Same tensors, semantics and
 * results as attn_chunk_bwd, but no workspace argument: the row dot products
 * go to a fixed 16 MiB array compiled into the library
 * (attn_chunk_bwd_noalloc_max_bytes()), which every GPU that loads the
 * library holds until the process exits; when the sequence-contiguous
 * operand copies of attn_chunk_bwd also fit, they are placed there too.
 *  - Limit: attn_chunk_bwd_min_workspace_size(q, k) must not exceed that
 *    size (B * Hq * Lq <= 4,194,304 query rows); larger problems return
 *    LSX_ERR_WORKSPACE and launch nothing.
 *  - The array is shared by every call on a device and keeps the last
 *    call's contents.  Each call rewrites what it reads (the row sums and
 *    statistics by its row-dot kernel; the fp32 dQ accumulator, when it fits,
 *    is cleared on the call's stream by cudaMemsetAsync, which allocates
 *    nothing).  Calls whose work overlaps on the GPU race on it: order them
 *    on one stream.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and caches it; make that
 *    first call before any stream capture.  With CUDA's default lazy module
 *    loading, that first call (or the first kernel of this library on the
 *    device) is also when the driver loads the library onto the device and
 *    reserves the 16 MiB: callers that may not take device memory after
 *    their start-up should make one call during start-up.
 *  - Allocates nothing (no cudaMalloc / cudaFree / allocating library call).
 * ---------------------------------------------------------------------- */
size_t attn_chunk_bwd_noalloc_max_bytes(void);
int attn_chunk_bwd_noalloc(const lsx_tensor* q, const lsx_tensor* k,
                           const lsx_tensor* v, const lsx_tensor* o,
                           const lsx_tensor* lse, const lsx_tensor* d_o,
                           int64_t q_off, int64_t kv_off, int causal,
                           float scale, const lsx_tensor* dq,
                           const lsx_tensor* dk, const lsx_tensor* dv,
                           int accumulate, lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_chunked_fwd / attn_chunked_bwd -- a whole sequence [B, H, N, D] split
 * into chunks of chunk_len rows, every (query chunk, key chunk) pair that the
 * mask leaves visible computed in ONE persistent launch whose CTAs take
 * work items from a longest-first causal schedule (DistFlashAttn, core
 * concepts: load-balanced scheduling; here the workers are the SMs).
 * chunk_len is validated (a positive multiple of 128) but is not a kernel
 * boundary: a work item walks the key tiles of consecutive chunks without
 * stopping, carrying one online softmax across the chunk edges, which equals
 * computing each chunk pair's partial and combining the partials with
 * attn_merge in that order (the merge is associative: Lean Attention
 * abstract).  Same dtypes as the chunk calls.
 *
 * Forward, split rows: when the query pairs (256 rows each) number fewer than
 * the SMs (few heads, long rows) and the rows are bf16 with D = 64 or 128,
 * every pair's visible key tiles are cut into pieces (about four pieces of
 * work per SM, at most 32 pieces per row).  Each piece writes its
 * normalised partial (fp32 O, LSE) to the workspace, and one more kernel
 * combines each row's pieces by the LSE-weighted merge (the stream-K style
 * split of the Lean Attention abstract; the result equals the unsplit one up
 * to fp32 rounding of the merge).  attn_chunked_fwd_workspace_size counts
 * those partials (for the current device's SM count); a workspace only as
 * large as attn_chunk_fwd_workspace_size, or none, runs the unsplit launch.
 * Otherwise the forward workspace holds the key-contiguous copy of V (as
 * attn_chunk_fwd).
 *
 * Backward, split key columns: its work items are (batch, kv head, key
 * tile), each walking the query tiles that see the key tile for every head
 * of the group.  When those items number fewer than the SMs (bf16, D = 64
 * or 128, not in deterministic mode), each item's steps are cut into pieces
 * (about four pieces of work per SM, at most 32 per item); every piece adds
 * its dQ contributions as usual and writes partial fp32 dK, dV to the
 * workspace, which one more kernel sums per key row (the result equals the
 * unsplit one up to fp32 rounding of the sums).
 * attn_chunked_bwd_workspace_size counts those partials; a workspace only as
 * large as attn_chunk_bwd_workspace_size runs the unsplit launch.
 * ---------------------------------------------------------------------- */
size_t attn_chunked_fwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k,
                                       int64_t chunk_len, int causal);
int attn_chunked_fwd(const lsx_tensor* q, const lsx_tensor* k,
                     const lsx_tensor* v, int64_t chunk_len, int causal,
                     float scale, const lsx_tensor* o, const lsx_tensor* lse,
                     void* workspace, size_t workspace_bytes,
                     lsx_stream_t stream);
size_t attn_chunked_bwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k,
                                       int64_t chunk_len, int causal);
int attn_chunked_bwd(const lsx_tensor* q, const lsx_tensor* k,
                     const lsx_tensor* v, const lsx_tensor* o,
                     const lsx_tensor* lse, const lsx_tensor* d_o,
                     int64_t chunk_len, int causal, float scale,
                     const lsx_tensor* dq, const lsx_tensor* dk,
                     const lsx_tensor* dv, void* workspace,
                     size_t workspace_bytes, lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_decode -- one query token per sequence against a long key/value
 * cache split into chunks of chunk_len keys; each chunk yields a partial
 * (O, LSE) and the partials are tree-reduced (Tree Attention abstract;
 * Lean Attention abstract: split-KV decode with a parallel reduction).
 *   q [B, Hq, 1, D] bf16; kc, vc [B, Hkv, N, D] bf16 (Hq / Hkv in
 *   {1, 2, 4, 8}); o [B, Hq, 1, D] bf16 or f32; lse [B, Hq, 1, 1] f32.
 * The query sees every key (no mask).  D == 128.
 * Workspace: attn_decode_workspace_size bytes (the per-chunk partials).
 * ---------------------------------------------------------------------- */
size_t attn_decode_workspace_size(const lsx_tensor* q, const lsx_tensor* kc,
                                  int64_t chunk_len);
int attn_decode(const lsx_tensor* q, const lsx_tensor* kc,
                const lsx_tensor* vc, int64_t chunk_len, float scale,
                const lsx_tensor* o, const lsx_tensor* lse, void* workspace,
                size_t workspace_bytes, lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_decode_tree -- one decode step for B branches of a tree of sequences
 * that share a prefix (Tree Attention page, related work: DeFT, tree-
 * structured decoding with KV-guided grouping): branch b's query attends to
 * the shared prefix followed by its own suffix.  The prefix cache is read
 * once per group of branches (up to 64 / G branches, G = Hq / Hkv), not once
 * per branch; the suffixes are read once each; all partials are merged in
 * one tree reduction.
 *   q [B, Hq, 1, D] bf16; pk, pv [1, Hkv, Np, D] bf16 (the shared prefix);
 *   sk, sv [B, Hkv, Ns, D] bf16 (the suffixes, Ns may be 0; NULL tensors
 *   are allowed when Ns == 0); o [B, Hq, 1, D] bf16 or f32; lse [B, Hq, 1, 1]
 *   f32.  Hq / Hkv in {1, 2, 4, 8}, D == 128, chunk_len a multiple of 128.
 * Workspace: attn_decode_tree_workspace_size bytes (the partials of both).
 * ---------------------------------------------------------------------- */
size_t attn_decode_tree_workspace_size(const lsx_tensor* q, const lsx_tensor* pk,
                                       const lsx_tensor* sk, int64_t chunk_len);
int attn_decode_tree(const lsx_tensor* q, const lsx_tensor* pk, const lsx_tensor* pv,
                     const lsx_tensor* sk, const lsx_tensor* sv, int64_t chunk_len,
                     float scale, const lsx_tensor* o, const lsx_tensor* lse, void* workspace,
                     size_t workspace_bytes, lsx_stream_t stream);

/* ------------------------------------------------------------------------
 * Status, diagnostics and host-side helpers.
 * ---------------------------------------------------------------------- */

/* Synchronises `stream`, returns the current device's status word (LSX_OK or
 * e.g. LSX_ERR_TIMEOUT) and clears it. */
int lsx_sync_status(lsx_stream_t stream);

/* Static string for a status code (never NULL). */
const char* lsx_status_string(int code);

/* Upper bound, in nanoseconds, of every device-side wait on an mbarrier
 * before the kernel gives up, records LSX_ERR_TIMEOUT and exits.  0 restores
 * the default (10 s).  Process-wide; affects launches made after the call. */
void lsx_set_wait_limit_ns(uint64_t ns);

/* Backward reduction order.  on == 0 (the default): for bf16 inputs one kernel
 * computes dK, dV and dQ together and adds each key tile's contribution to
 * dQ into an fp32 accumulator with reduce-adds (TMA bulk or vector atomic),
 * performed at L2 in no fixed order, so dQ's rounding
 * depends on the order in which those adds land (results agree with the
 * deterministic mode within the documented tolerance, not bit for bit).
 * on != 0: dQ is computed by a second kernel in which every dQ row is owned
 * by one thread block, and repeated calls on the same inputs give identical
 * bytes (slower: the score tiles are rebuilt a second time).  dK and dV are
 * identical between calls in both modes.  Process-wide; affects calls made
 * after it. */
void lsx_set_deterministic(int on);

/* Launches one block that waits on an mbarrier nothing will ever complete,
 * under the current wait limit, so that callers can check that a bounded wait
 * ends and reports LSX_ERR_TIMEOUT through lsx_sync_status (no fault, no
 * hang). */
int lsx_selftest_bounded_wait(lsx_stream_t stream);

/* Host-only: simulate the forward work schedule that attn_chunked_fwd would
 * use for [B, H, N] with chunk_len and causal, on n_workers persistent
 * workers, with each work item costed by its visible key tiles.  Writes
 * makespan (max tiles on one worker), the ideal (total / n_workers, rounded
 * up) and the total into out[0..2].  host pointers. */
int lsx_schedule_stats(int64_t B, int64_t H, int64_t N, int64_t chunk_len,
                       int causal, int n_workers, int64_t* out);

/* Device-side record of the balanced causal schedule (DistFlashAttn, core
 * concepts: load-balanced scheduling removes the idle time of the workers
 * that finish early; here the workers are the SMs of one GPU).  While a trace
 * buffer is set, every launch of a persistent tensor-core kernel (the
 * forward, the fused or the dK/dV backward, the deterministic dQ kernel)
 * appends one record to it, written by the kernel itself:
 *   uint64 words [0] kernel id (0 forward, 1 dK/dV, 2 dQ, 12 fused dK/dV/dQ),
 *   [1] G = CTAs in the launch, [2] work items in the launch, then for each
 *   CTA c: [3 + 3c] its %globaltimer (ns) before its first item, [4 + 3c]
 *   after its last item (every role done), [5 + 3c] the items it ran.
 * The SM idle fraction of a launch is 1 - sum_c (end_c - start_c) /
 * (G * (max end - min start)).
 *   buf: DEVICE memory owned by the caller, 8-byte aligned, or NULL to stop
 *   tracing; bytes: its size.  A launch whose record would not fit is not
 *   traced (not an error).  Enabling resets the fill level to 0.
 * lsx_trace_used returns the bytes handed out to records since the last
 * lsx_trace_enable (read the buffer after the launches have completed).
 * Process-wide and for diagnosis only: costs one predicated branch per CTA
 * when off, two %globaltimer reads and 24 bytes per CTA when on. */
int lsx_trace_enable(void* buf, size_t bytes);
size_t lsx_trace_used(void);

/* Library version string, e.g. "lsx 0.1 sm_103a". */
const char* lsx_version(void);

/* Per-kernel timing.  While enabled, every kernel launch of the library is
 * bracketed by a pair of CUDA events recorded on the launching stream (the
 * events are created by the library on first use; no device memory).
 * lsx_timing_report synchronises those events and writes, for each kernel
 * that ran since the last reset, one line "name launches total_ms\n" into
 * buf (host memory, NUL-terminated, truncated to n bytes); it returns the
 * number of kernels reported or a negative status.  lsx_timing_reset drops
 * the recorded events.  Process-wide; not meant for concurrent callers. */
int lsx_timing_enable(int on);
int lsx_timing_report(char* buf, size_t n);
int lsx_timing_reset(void);

#ifdef __cplusplus
}
#endif
#endif /* LSX_H */
