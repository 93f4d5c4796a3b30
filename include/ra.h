/*
 * ra.h -- C ABI of the GB300 ring-attention forward library (libra.so).
 *
 * What the library computes (ring attention, forward):
 *   Q, K and V are split along the sequence into N shards.  Shard p keeps its
 *   query block; at ring step t = 0..N-1 it meets the K/V block of shard
 *   r = (p - t) mod N ("device i -> i+1" rotation: "3.6 Distributed Training II",
 *   section "Ring Attention"; the Q&A page "Explain ring attention ...", section
 *   "The ring").  Each block is folded into a running max m, running sum l and
 *   output accumulator o by the online-softmax update of "Module 23: Distributed
 *   Training", section "The Math: One Block at a Time"; at the end O = o / l.
 *   Causal attention skips blocks strictly in the future of a query tile and
 *   masks the rest key by key on global positions (Module 23, "Exact by
 *   Construction"); the diagonal is kept (key position <= query position).
 *
 *   One GPU runs all N shards: the ring rotation becomes the order in which
 *   each query tile visits K/V tiles.  There are no inter-GPU transfers.
 *
 * Tensor conventions shared by every entry point:
 *   - Q, O:   [B, Hq,  S, d] row-major, contiguous.
 *   - K, V:   [B, Hkv, S, d] row-major, contiguous.
 *   - LSE:    [B, Hq,  S] float32, natural-log log-sum-exp of the scaled,
 *             masked scores of each row (the pages return O only; the LSE is
 *             what lets partial results be merged).
 *   - The S axis is in LAYOUT ORDER: shard p occupies rows [p*S/N, (p+1)*S/N),
 *     and row p*S/N + i holds the token at natural position pos(p, i):
 *       contiguous: p*S/N + i
 *       striped:    i*N + p                 (Module 23, "The Causal Imbalance --
 *                                            and the Striped Fix")
 *       zigzag:     with c = S/(2N): i < c ? p*c + i : (2N-1-p)*c + (i - c)
 *                   (reading of "the same idea, paired up block-by-block": chunk p
 *                   paired with chunk 2N-1-p)
 *     ra_layout_perm converts natural order <-> layout order.
 *   - GQA: query head h reads key/value head h / (Hq/Hkv).
 *   - Scores are s = scale * q.k with scale = 1/sqrt(d) unless given.
 *
 * Ownership: the caller owns every device buffer passed in.  A plan owns its
 * host tables, its device work tables (whole forward, one per ring step, backward),
 * its device status word, a stream for its own allocations and frees, three CUDA
 * events for ra_ring_fwd, and one event per stream its kernels were launched on;
 * ra_fwd, ra_fwd_step, ra_ring_rotate, ra_ring_fwd, ra_bwd, ra_merge_partials and
 * ra_layout_perm allocate no device memory ("allocates nothing" below: the first
 * launch of a plan on a stream it has not used creates that stream's event) and are
 * asynchronous on the given stream (a cudaStream_t passed as void*; NULL = legacy
 * default).
 *
 * Errors: every call returns an ra_status; on failure ra_last_error() returns a
 * thread-local message.  Arguments are checked before anything is launched.
 * Every device buffer must be memory of the CURRENT device (or managed memory)
 * and every stream must belong to it: the kernels run on the current device, so
 * a buffer of another device or a host pointer is rejected with
 * RA_ERR_INVALID_ARG before any launch (RA_ERR_NO_DEVICE when no device exists).
 * Uneven shards are rejected, never padded (Module 23, "Common Pitfalls":
 * reject uneven shards rather than silently bias the result).
 */
#ifndef RA_H_
#define RA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, uneven shards */
  RA_ERR_UNSUPPORTED = 2,  /* valid problem outside what the kernels handle      */
  RA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed               */
  RA_ERR_TIMEOUT = 4,      /* a device-side wait exceeded its budget (~1 s)      */
  RA_ERR_NO_DEVICE = 5,    /* the plan has no device state (no GPU at plan time) */
  RA_ERR_BOUNDS = 6        /* debug build only: a kernel's bounds check failed    */
} ra_status;

typedef enum {
  RA_LAYOUT_CONTIGUOUS = 0,
  RA_LAYOUT_STRIPED = 1,
  RA_LAYOUT_ZIGZAG = 2
} ra_layout;

typedef enum {
  RA_DTYPE_F32 = 0,   /* float32 Q/K/V/O; SIMT kernel, d <= 128              */
  RA_DTYPE_BF16 = 1   /* bfloat16 Q/K/V/O; tensor-core kernel, d == 128      */
} ra_dtype;

/* One attention problem.  All sizes are element counts. */
typedef struct {
  int64_t batch;     /* B  >= 1                                            */
  int64_t seq;       /* S  >= 1, multiple of n_shards (2*n_shards: zigzag) */
  int32_t heads_q;   /* Hq >= 1, multiple of heads_kv                      */
  int32_t heads_kv;  /* Hkv >= 1                                           */
  int32_t head_dim;  /* d: 128 for BF16; 1..128 for F32                    */
  int32_t n_shards;  /* N >= 1                                             */
  int32_t layout;    /* ra_layout                                          */
  int32_t causal;    /* 0 or 1                                             */
  int32_t dtype;     /* ra_dtype                                           */
  float scale;       /* score scale; 0 selects 1/sqrt(head_dim)            */
} ra_problem;

typedef struct ra_plan_s* ra_plan_t;

/*
 * ra_plan -- validate a problem and build its ring schedule.
 * Builds, on the host, the per-shard tile classification (FULL / PARTIAL / SKIP,
 * see ra_plan_tile_counts) and, for BF16 problems, the work lists of the
 * tensor-core kernels: the whole forward (ra_fwd), one list per ring step
 * (ra_fwd_step), the gathered forward (ra_fwd_gathered) and the two backward
 * passes (ra_bwd), each in longest-first order with key/value heads grouped.  It
 * also picks each kernel's schedule: synchronised rounds when one key/value head's
 * K and V exceed 32 MiB, otherwise items handed out as CTAs free up.  When a CUDA
 * device is current, it uploads the work tables and allocates the plan's device
 * status word (stream-ordered, on a stream of the plan's own; the call returns once
 * they are in place), and creates the three events ra_ring_fwd orders its streams
 * with.  Without a
 * device the plan is host-only: tile counts work, the compute calls return
 * RA_ERR_NO_DEVICE.
 * *out receives the plan; release it with ra_plan_destroy.
 * Errors: RA_ERR_INVALID_ARG (null pointers, sizes < 1, S % N, zigzag S % 2N,
 * Hq % Hkv, bad enum), RA_ERR_UNSUPPORTED (BF16 with d != 128, F32 with d > 128,
 * more than 2^31 rows, more than 32767 shards; a plan too large to build on the
 * host: N^2 x query tiles per shard above 2^30, BF16 work lists above 2^27
 * entries, or a host allocation that failed), RA_ERR_CUDA (device upload failed).
 */
ra_status ra_plan(const ra_problem* prob, ra_plan_t* out);

/* Release a plan and its device memory.  NULL is accepted.  It does not wait:
 * kernels queued with this plan may still read its tables, so the plan records
 * an event on every stream it launched on (after its latest launch there), and
 * the frees of its device memory are queued in stream order behind those events
 * only (cudaFreeAsync on the plan's own stream; the plan allocated its tables
 * with cudaMallocAsync).  Other streams' work and other plans' kernels are not
 * waited for.  Do not use the plan after this call.  It does not clear a pending
 * CUDA error. */
ra_status ra_plan_destroy(ra_plan_t plan);

/*
 * ra_plan_tile_counts -- per-shard causal tile classification of the schedule.
 * For one (batch entry, query head), counts over all N ring steps the pairs
 * (128-row query tile of shard p, 128-row key tile of the block met at step t)
 * that are FULL (every (q,k) pair causal), PARTIAL (some) or SKIP (none),
 * following Module 23's per-device causal work count ("The Causal Imbalance")
 * at tile granularity.  The last tile of a shard may be shorter than 128.
 * Non-causal problems count every tile FULL.  full, partial and skip are
 * caller-owned host arrays of n_shards int64 each (any may be NULL).
 */
ra_status ra_plan_tile_counts(ra_plan_t plan, int64_t* full, int64_t* partial, int64_t* skip);

/*
 * ra_fwd -- ring-attention forward on the plan's problem.
 * q, k, v: device pointers, layout order, dtype of the plan, 16-byte aligned.
 * Fused mode (o_parts == lse_parts == NULL):
 *   o   [B, Hq, S, d] in the plan's dtype (required);
 *   lse [B, Hq, S] float32 (may be NULL).
 * Partials mode (o_parts and lse_parts non-NULL, o == lse == NULL):
 *   o_parts   [N, B, Hq, S, d] float32 and lse_parts [N, B, Hq, S] float32;
 *   entry t of a row of shard p is attention of that row over the key block of
 *   shard (p - t) mod N alone, normalised by its own sum; a block with no causal
 *   key gives O_t = 0, LSE_t = -inf.  ra_merge_partials combines them.
 * Asynchronous on stream; allocates nothing.  A device-side wait that runs out
 * of budget makes the kernel return early and sets the plan's status word;
 * ra_sync_status reports it.  Calls that share a plan must not overlap on the
 * GPU (the plan's device words hold the status and the work-item counter).
 * Errors: RA_ERR_INVALID_ARG (null/misaligned pointers, mixed modes),
 * RA_ERR_NO_DEVICE, RA_ERR_CUDA (launch failure).
 */
ra_status ra_fwd(ra_plan_t plan, const void* q, const void* k, const void* v,
                 void* o, float* lse, float* o_parts, float* lse_parts, void* stream);

/*
 * ra_fwd_step -- one ring step for every shard, run as the device holding the shard
 * runs it: each shard attends to the K/V block it holds at that step.
 * At step t shard p holds the block that started on shard (p - t) mod N, passed
 * on one device per step (device i -> i+1: "3.6 Distributed Training II",
 * section "Ring Attention"; the Q&A page, section "The ring").
 * step: t in [0, N).
 * q: [B, Hq, S, d] in layout order.
 * k_blk, v_blk: [B, Hkv, S, d] receive buffers.  The rows of shard p, [p*S/N, (p+1)*S/N),
 *   hold the block shard p holds at step t: K/V themselves at t = 0, then what t
 *   calls of ra_ring_rotate have passed along.
 * o_part [B, Hq, S, d] float32 and lse_part [B, Hq, S] float32 receive the
 *   attention of every row over that block alone, with the conventions of
 *   ra_fwd's partials mode: normalised by its own sum; O_t = 0 and LSE_t = -inf
 *   where the block has no causal key.  The result equals entry t of ra_fwd's
 *   partials.
 * Device pointers in the plan's dtype (o_part/lse_part float32), 16-byte aligned.
 * Asynchronous on stream; allocates nothing; the plan holds one work list per step.
 * Calls that share a plan must not overlap on the GPU.
 * Errors: RA_ERR_INVALID_ARG (step out of range, null/misaligned pointers),
 * RA_ERR_NO_DEVICE, RA_ERR_CUDA.
 */
ra_status ra_fwd_step(ra_plan_t plan, int32_t step, const void* q, const void* k_blk,
                      const void* v_blk, float* o_part, float* lse_part, void* stream);

/*
 * ra_ring_rotate -- the ring's exchange, in which every shard passes its K/V block on
 * to the next: for each [S, d] matrix of K and V ([B, Hkv, S, d], plan dtype), the
 * rows of shard (p + 1) mod N in the destination receive the rows of shard p in the
 * source (device i -> i+1; "3.6 Distributed Training II", "Ring Attention").
 * The copies are copy-engine transfers, two per tensor (strided over B*Hkv), so
 * they can run on a second stream while a forward kernel occupies every SM.  That
 * is one GPU's stand-in for the send/receive that overlaps compute between devices.
 * k_src, v_src, k_dst, v_dst: device pointers.  A destination must not overlap its
 * source or the other destination.  Asynchronous on stream; allocates nothing.
 * Errors: RA_ERR_INVALID_ARG (null pointers, overlap), RA_ERR_NO_DEVICE, RA_ERR_CUDA.
 */
ra_status ra_ring_rotate(ra_plan_t plan, const void* k_src, const void* v_src, void* k_dst,
                         void* v_dst, void* stream);

/*
 * ra_ring_fwd -- the explicit ring driver.  It runs N calls of ra_fwd_step on
 * `stream`.  While step t computes, ra_ring_rotate passes the block of step t on
 * to the receive buffer of step t+1, on `comm_stream`: the overlap of
 * communication with compute that "3.6 Distributed Training II", "Ring
 * Attention", describes.  Then it merges the N partials with ra_merge_partials
 * (Module 23, "The Math: One Block at a Time": the fold is order independent).
 * q, k, v: as for ra_fwd.
 * o [B, Hq, S, d] (plan dtype) and lse [B, Hq, S] float32 (may be NULL) receive
 *   the fused result.
 * k_buf, v_buf: caller-owned scratch, two receive buffers each: [2, B, Hkv, S, d]
 *   in the plan's dtype.  They must not overlap each other or K/V.  May be NULL
 *   when N == 1.
 * o_parts [N, B, Hq, S, d] and lse_parts [N, B, Hq, S]: caller-owned float32
 *   scratch for the per-step partials; they hold them after the call.
 * stream: the compute stream.  comm_stream: the rotation stream; it may equal
 *   stream, and then nothing overlaps.  The driver orders both streams with three
 *   events that the plan owns.  Work already queued on stream comes before the
 *   rotations; later work on stream comes after the driver's work on both streams.
 * Asynchronous; allocates nothing.  Calls that share a plan must not overlap.
 * Errors: as ra_fwd_step, ra_ring_rotate and ra_merge_partials.
 */
ra_status ra_ring_fwd(ra_plan_t plan, const void* q, const void* k, const void* v, void* o,
                      float* lse, void* k_buf, void* v_buf, float* o_parts, float* lse_parts,
                      void* stream, void* comm_stream);

/*
 * ra_bwd -- gradients of the ring-attention forward (dQ, dK, dV from dO).
 * The pages present ring attention as a way to train on long sequences (the
 * activations of every layer are kept for the backward pass: "3.6 Distributed
 * Training II", section "Ring Attention") but print no backward pass; this one
 * differentiates the forward's definition O = softmax(scale * Q K^T + M) V:
 *   P = exp(scale * Q K^T + M - LSE)   (recomputed from the forward's LSE)
 *   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D = rowsum(dO * O),
 *   dQ = scale * dS K,  dK = scale * dS^T Q,
 * with a key/value head's dK and dV summed over the query heads that read it.
 * The work follows the ring: a query tile of shard p meets the key blocks of
 * shards (p - t) mod N (as in the forward); a key block of shard r meets the
 * queries of shard (r + t) mod N at step t, so its gradients gather where the
 * block travels.
 * q, k, v, o, dout (dO): as for ra_fwd (layout order, plan dtype); o and lse
 *   are the forward's outputs for the same q, k, v.
 * dq [B, Hq, S, d], dk and dv [B, Hkv, S, d]: outputs, plan dtype.
 * scratch: caller-owned float32 device buffer of ra_bwd_scratch_size bytes (per
 *   query row LSE * log2(e) and D, in blocks of 64 rows of one shard).
 * Device pointers, 16-byte aligned.  Asynchronous on stream; allocates nothing.
 * A device-side wait that runs out of budget is reported by ra_sync_status.
 * Calls that share a plan must not overlap on the GPU.
 * Errors: RA_ERR_INVALID_ARG (null/misaligned pointers), RA_ERR_NO_DEVICE,
 * RA_ERR_CUDA.
 */
ra_status ra_bwd(ra_plan_t plan, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dout, void* dq, void* dk, void* dv, float* scratch,
                 void* stream);

/*
 * ra_bwd_scratch_size -- bytes of the scratch buffer ra_bwd needs for this plan:
 * 512 bytes per 64-row block of every (batch, query head, shard), about
 * 8 * B * Hq * S bytes.  Host only.  Errors: RA_ERR_INVALID_ARG (null arguments).
 */
ra_status ra_bwd_scratch_size(ra_plan_t plan, int64_t* bytes);

/*
 * ra_allgather_kv -- the all-gather of the all-gather variant of context parallelism:
 * every device gathers the K/V blocks of all shards instead of passing them around
 * a ring ("3.6 Distributed Training II", section "Ring Attention": the Llama 3
 * paper's context parallelism for long-context training, with an all-gather of K/V
 * rather than a ring).  One GPU keeps one gathered copy: k_all, v_all
 * [B, Hkv, S, d] receive K and V in NATURAL order (row = token position).
 * k, v: [B, Hkv, S, d] in layout order.  Device pointers, plan dtype, 16-byte
 * aligned; a destination must not overlap its source or the other destination.
 * Asynchronous on stream; allocates nothing.
 * Errors: RA_ERR_INVALID_ARG (null/misaligned pointers, overlap), RA_ERR_NO_DEVICE,
 * RA_ERR_CUDA.
 */
ra_status ra_allgather_kv(ra_plan_t plan, const void* k, const void* v, void* k_all, void* v_all,
                          void* stream);

/*
 * ra_fwd_gathered -- the forward of the all-gather variant: every query row of
 * shard p attends over the gathered K/V in one step, causal by position (the keys
 * at or before its own position; Module 23, "Exact by Construction").  The result
 * is the same attention as ra_fwd; only the data movement differs.
 * q: [B, Hq, S, d] in layout order; k_all, v_all: [B, Hkv, S, d] in natural order
 * (ra_allgather_kv); o [B, Hq, S, d] (plan dtype) and lse [B, Hq, S] float32 (may be
 * NULL) in layout order.  Device pointers, 16-byte aligned.  Asynchronous on stream;
 * allocates nothing.  Calls that share a plan must not overlap on the GPU.
 * Errors: RA_ERR_INVALID_ARG (null/misaligned pointers), RA_ERR_NO_DEVICE, RA_ERR_CUDA.
 */
ra_status ra_fwd_gathered(ra_plan_t plan, const void* q, const void* k_all, const void* v_all,
                          void* o, float* lse, void* stream);

/*
 * ra_ulysses_a2a -- DeepSpeed-Ulysses' all-to-all for N devices (the Q&A page
 * "Explain ring attention ...", section "Related approaches": split by attention
 * heads with an all-to-all instead of a ring).  Each device starts with its
 * sequence shard of every head; the exchange hands device p' every token, by
 * position, of heads p'*H/N .. (p'+1)*H/N - 1, where it runs ordinary attention over
 * the whole sequence (ra_fwd with a plan of batch N*B, H/N heads, one shard); the
 * reverse exchange returns O (and the LSE) to the sequence shards.
 * direction 0 (sequence -> heads): src [B, H, S, row] in layout order (shard p =
 *   rows [p*S/N, (p+1)*S/N)), dst [N, B, H/N, S, row] (device p', natural order).
 * direction 1 (heads -> sequence): src [N, B, H/N, S, row], dst [B, H, S, row].
 * row_bytes: 256 (d = 128 bf16) or 4 (the float32 LSE).  heads: H, a multiple of N.
 * Device pointers, 16-byte aligned, not overlapping.  Asynchronous; allocates nothing.
 * Errors: RA_ERR_INVALID_ARG (uneven shards, heads % N, direction, pointers),
 * RA_ERR_UNSUPPORTED (row_bytes, more than 2^31-1 rows), RA_ERR_CUDA.
 */
ra_status ra_ulysses_a2a(int32_t direction, int32_t layout, int64_t seq, int32_t n_shards,
                         int64_t batch, int32_t heads, int32_t row_bytes, const void* src, void* dst,
                         void* stream);

/*
 * ra_merge_partials -- exact combination of partial attention results.
 * For each of `rows` rows: LSE = ln sum_t e^(LSE_t), O = sum_t e^(LSE_t - LSE) O_t
 * (order independence of the online-softmax fold, Module 23, "The Math: One
 * Block at a Time").  Parts with LSE_t = -inf are ignored; a row whose parts are
 * all -inf gets O = 0 and LSE = -inf.
 * o_parts [n_parts, rows, d] float32, lse_parts [n_parts, rows] float32, o [rows, d]
 * in o_dtype (F32 or BF16, round-to-nearest-even), lse [rows] float32 or NULL.
 * Device pointers, 16-byte aligned.  Asynchronous on stream; allocates nothing.
 * Errors: RA_ERR_INVALID_ARG (sizes < 1, d > 1024, null/misaligned pointers),
 * RA_ERR_CUDA.
 */
ra_status ra_merge_partials(int32_t n_parts, int64_t rows, int32_t d,
                            const float* o_parts, const float* lse_parts,
                            void* o, int32_t o_dtype, float* lse, void* stream);

/*
 * ra_layout_perm -- move whole rows between natural order and layout order.
 * src and dst are [rows_outer, seq, row_bytes] (e.g. Q as [B*Hq, S, d*2] bytes).
 * inverse == 0: dst[o, j] = src[o, pos(j)]   (natural -> layout order)
 * inverse != 0: dst[o, pos(j)] = src[o, j]   (layout -> natural order)
 * with pos the layout map above.  row_bytes must be a multiple of 4; pointers
 * 16-byte aligned; src and dst must not overlap.  Asynchronous; allocates nothing.
 * Errors: RA_ERR_INVALID_ARG (uneven shards, bad sizes, overlap, alignment),
 * RA_ERR_UNSUPPORTED (seq above 2^31-1, n_shards above 32767, more than 2^63-1 bytes),
 * RA_ERR_CUDA.
 */
ra_status ra_layout_perm(int32_t layout, int64_t seq, int32_t n_shards, int32_t inverse,
                         int64_t rows_outer, int32_t row_bytes,
                         const void* src, void* dst, void* stream);

/*
 * ra_layout_index -- host helper: pos_out[j] = natural position of layout row j,
 * for j in [0, seq).  pos_out is a caller-owned host array of seq int64.
 * Errors: RA_ERR_INVALID_ARG (uneven shards, null pointer, bad layout).
 */
ra_status ra_layout_index(int32_t layout, int64_t seq, int32_t n_shards, int64_t* pos_out);

/*
 * ra_sync_status -- synchronize `stream`, then read and clear the plan's device
 * status word.  Returns RA_ERR_TIMEOUT if a kernel launched with this plan gave
 * up on a device-side wait since the last call, RA_ERR_BOUNDS if (in the debug
 * build, libra_debug.so, compiled with RA_DEBUG_BOUNDS) one of its bounds checks
 * failed, RA_ERR_CUDA on a CUDA error, RA_OK otherwise.
 */
ra_status ra_sync_status(ra_plan_t plan, void* stream);

/*
 * ra_fwd_static -- the bf16 fused forward for callers that cannot allocate.
 * The pages have no counterpart to this entry point; it exists for callers that
 * must not allocate device memory at run time (code running under an allocator
 * or memory pool it may not bypass, or with a device footprint fixed at load
 * time) and therefore cannot create a plan, since ra_plan allocates the work
 * table and status word.  It computes exactly what ra_fwd computes in fused mode
 * for a bf16, head_dim 128 problem, without a plan and without allocating:
 * no cudaMalloc, cudaFree or other allocating routine is called.
 *   - Scratch: the work table and status word live in one file-scope device
 *     array of 4 MiB + 256 B, held on every GPU that loads the library until the
 *     process exits.  Problems needing more than 131072 work items (one item per
 *     pair of 128-row query tiles; e.g. 1M tokens x 32 query heads is exactly
 *     131072), or more than 2^30 (item, ring step) pairs to cost, are rejected
 *     with RA_ERR_UNSUPPORTED.
 *   - Set-up: the first call on a device (with that device current) looks up the
 *     array's device address (a host-side runtime query, made once per device).
 *   - Sharing: every call reuses the array; the status word is cleared at the
 *     start of each call.  Calls whose kernels overlap on the GPU race on the
 *     array and must not be issued; calls from several host threads are
 *     serialised on the host.  Device-side wait timeouts are recorded in the
 *     array's status word, which ra_fwd_static_status reports.
 * prob: the problem (dtype RA_DTYPE_BF16, head_dim 128).  q, k, v, o, lse: as for
 * ra_fwd in fused mode (lse may be NULL), device pointers, 16-byte aligned.
 * Asynchronous on stream.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED (dtype, head_dim, size),
 * RA_ERR_NO_DEVICE, RA_ERR_CUDA.
 */
ra_status ra_fwd_static(const ra_problem* prob, const void* q, const void* k, const void* v,
                        void* o, float* lse, void* stream);

/*
 * ra_fwd_static_status -- the device-wait status of the latest ra_fwd_static
 * call on the current device.  Like ra_fwd_static, no counterpart on the pages.
 * Synchronizes `stream` (the stream that call ran on), then reads and clears the
 * status word in the static array: RA_ERR_TIMEOUT if that call's kernel gave up
 * on a device-side wait (its O/LSE are then incomplete), RA_ERR_BOUNDS if a
 * bounds check of the debug build failed, RA_OK otherwise or when ra_fwd_static
 * has not run on this device.  It allocates nothing.  The next ra_fwd_static call
 * clears the word, so read it before issuing another.
 * Errors: RA_ERR_TIMEOUT, RA_ERR_BOUNDS, RA_ERR_NO_DEVICE, RA_ERR_CUDA.
 */
ra_status ra_fwd_static_status(void* stream);

/*
 * ra_wait_selftest -- check the failure-detection path of the tensor-core kernels.
 * Not a step of the method.  Every mbarrier wait in the tensor-core kernels gives
 * up after about one second, records a bit in a device status word and lets its
 * kernel return, so that a handshake that never comes ends in RA_ERR_TIMEOUT
 * (ra_sync_status) instead of a hung GPU.  This call runs that wait routine once
 * in a one-warp kernel against an mbarrier that nothing ever arrives on.
 * *status_out (host) receives the status word the wait left: 2 (the MMA-side bit
 * of ra_sync_status's message) when it gave up as designed, 0 if it never did.
 * Later launches in the same context are unaffected.
 * Synchronous, on the legacy default stream of the current device; it takes
 * about one second.  It allocates one 4-byte device word and frees it.
 * Errors: RA_ERR_INVALID_ARG (null status_out), RA_ERR_NO_DEVICE, RA_ERR_CUDA.
 */
ra_status ra_wait_selftest(uint32_t* status_out);

/* Thread-local message describing the last failure on this thread ("" if none). */
const char* ra_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
