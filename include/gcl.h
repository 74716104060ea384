/*
 * gcl.h -- C ABI of the GB300 chunked gated linear attention library (libgcl).
 *
 * The library computes the chunkwise Map-Reduce-Map prefill of two recurrences
 * over varlen batches addressed by cu_seqlens:
 *
 *   GDN  S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   KDA  S_t = (I - beta_t k_t k_t^T) Diag(a_t) S_{t-1} + beta_t k_t v_t^T
 *        o_t = S_t^T (scale q_t),  alpha_t = exp(g_t),  a_t = exp(g_t) (per key channel)
 *
 * Sources: HA-NPU paper "Empowering Hybrid Attention Models on NPUs"
 * (section 2.1: fixed-size recurrent state per head, chunkwise Map-Reduce-Map;
 * section 4: head-level mapping and column-wise split of tail heads;
 * section 5: chunk-first in-place state update, W = A^-1 K and the grouped
 * GEMMs KS, QS, KK^T, QK^T) and the FLA RFC "[RFC] Add Graph Capture Support
 * for FLA Prefill and Training Paths on Ascend NPUs" (section "Core design":
 * fixed capacity T_max / N_max / BT / NT_max, the [-1, 0] sentinel, device-side
 * metadata, the static buffer contract; section "API proposal":
 * max_num_seqs, chunk_indices, chunk_offsets, fail clearly, no silent fallback).
 *
 * Conventions shared by every entry point
 *  - Every pointer named "device" is a CUDA device pointer owned by the caller.
 *    The library never allocates, frees, synchronises or creates graphs.
 *  - `stream` is a cudaStream_t passed as an opaque pointer (NULL = legacy
 *    default stream).  All work is enqueued on it; calls return before the GPU
 *    finishes.  Launch configurations depend only on the sizes given here, never
 *    on device data, so every call may be captured into a CUDA graph and
 *    replayed after the caller updates its buffers in place.
 *  - Host-checkable errors (NULL where a pointer is required, unsupported sizes
 *    or dtypes, misaligned pointers) return a non-zero gcl_status_t before any
 *    work is enqueued; nothing falls back to another implementation.
 *    gcl_last_error() gives a one-line reason (per calling thread).
 *  - Data-dependent errors are reported through `dev_status`, a device int32:
 *    chunk_meta_build writes 0 (ok) or a GCL_DEV_* code; the compute entry
 *    points read it first and do nothing when it is non-zero.  The caller reads
 *    it after its own synchronisation.
 *  - Layouts are token-major and row-major (contiguous):
 *      q, k [T_max, H, K];  v, o [T_max, H, V];  beta [T_max, H];
 *      g [T_max, H] (GDN) or [T_max, H, K] (KDA), fp32 log-space gate (<= 0);
 *      states h0, ht, dht, dh0 [N_max, H, K, V] fp32.
 *    Token rows at or past cu_seqlens[N_max] are never read or written.
 */
#ifndef GCL_H
#define GCL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gcl_status {
    GCL_OK = 0,
    GCL_ERR_INVALID_ARG = 1,   /* NULL pointer, inconsistent or out-of-range size */
    GCL_ERR_UNSUPPORTED = 2,   /* size, dtype or chunk size this library does not implement */
    GCL_ERR_CAPACITY = 3,      /* a fixed capacity (workspace, scratch) is too small */
    GCL_ERR_CUDA = 4           /* a CUDA call failed (message in gcl_last_error) */
} gcl_status_t;

/* Device status word values (written by chunk_meta_build). */
#define GCL_DEV_OK 0
#define GCL_DEV_CU_DECREASING 1    /* cu_seqlens[n+1] < cu_seqlens[n] for some n        */
#define GCL_DEV_CU_NONZERO_START 2 /* cu_seqlens[0] != 0                                 */
#define GCL_DEV_CU_OVER_CAPACITY 3 /* cu_seqlens[N_max] > T_max                          */
#define GCL_DEV_BAD_RANGE 4        /* a compute kernel met an invalid sequence range      */
#define GCL_DEV_WAIT_TIMEOUT 5     /* a kernel gave up waiting on an async copy or MMA    */
#define GCL_DEV_OUT_OF_BOUNDS 6    /* debug build (GCL_DEBUG_BOUNDS): an index fell       */
                                   /* outside its buffer; the access was skipped          */

typedef enum gcl_dtype {
    GCL_F32 = 0,   /* q, k, v, beta, do, o in fp32; every internal product in fp32     */
    GCL_BF16 = 1,  /* q, k, v, beta, do, o in bf16; state and accumulation in fp32     */
    GCL_F16 = 2    /* q, k, v, beta, do, o in fp16; the GDN forward with K = V = 128,   */
                   /* bt = 64 on the tensor cores (fp16 MMA operands, fp32 state and   */
                   /* accumulation), every other product in fp32                      */
} gcl_dtype_t;

typedef void *gcl_stream_t;

/* One-line reason for the last non-OK status returned on this thread ("" if none). */
const char *gcl_last_error(void);

/* Name of a gcl_status_t or GCL_DEV_* value. */
const char *gcl_status_string(int32_t status);

/*
 * NT_max = ceil(t_max / bt) + n_max - 1: the most chunks any layout of at most
 * t_max tokens in at most n_max sequences can have (FLA RFC, "Core design /
 * Fixed-capacity execution").  Returns -1 for non-positive arguments.
 */
int64_t gcl_nt_max(int64_t t_max, int64_t n_max, int32_t bt);

/*
 * chunk_meta_build -- device-side chunk metadata (FLA RFC, "Core design /
 * Device-side metadata"; zero-length tail sequences from "Step 1").
 *
 *   cu_seqlens     device int32 [n_max + 1], non-decreasing, cu_seqlens[0] = 0,
 *                  cu_seqlens[n_max] <= t_max; zero-length sequences allowed.
 *   chunk_indices  device int32 [nt_max, 2] (out): row j = (n, i) for the i-th
 *                  chunk of sequence n, rows in sequence-major order; rows at or
 *                  past the live chunk count hold the sentinel [-1, 0].
 *   chunk_offsets  device int32 [n_max + 1] (out): exclusive prefix sum of the
 *                  per-sequence chunk counts ceil(len_n / bt); the last entry is
 *                  the live chunk count.
 *   seq_order      device int32 [n_max] (out, may be NULL): sequence indices
 *                  sorted by length, longest first (ties by index); the compute
 *                  kernels use it to start long sequences first.
 *   dev_status     device int32 [1] (out): GCL_DEV_OK, or the first failing check
 *                  in the order NONZERO_START, DECREASING, OVER_CAPACITY.  On
 *                  failure every row is the sentinel, every offset is 0 and
 *                  seq_order is the identity, so later kernels do no work.
 *   nt_max         must equal gcl_nt_max(t_max, n_max, bt).
 *
 * One kernel launch; no host synchronisation; graph-capturable.
 * Host errors: INVALID_ARG for NULL required pointers, n_max < 1, t_max < 1,
 * t_max >= 2^31, bt < 1 or nt_max mismatch.
 */
gcl_status_t chunk_meta_build(const int32_t *cu_seqlens, int32_t n_max, int64_t t_max,
                              int32_t bt, int64_t nt_max, int32_t *chunk_indices,
                              int32_t *chunk_offsets, int32_t *seq_order,
                              int32_t *dev_status, gcl_stream_t stream);

/*
 * chunk_meta_build_i64 -- chunk_meta_build for an int64 cu_seqlens (FLA RFC,
 * "Improve the common graph infrastructure": int32 and int64 cu_seqlens).
 *
 *   cu_seqlens     device int64 [n_max + 1], with the contract of chunk_meta_build.
 *   cu_seqlens32   device int32 [n_max + 1] (out): the same offsets narrowed to
 *                  int32 (exact: a valid cu_seqlens lies in [0, t_max], t_max < 2^31),
 *                  or all zeros when a check fails.  Pass it as cu_seqlens to the
 *                  compute calls, whose arguments are int32.
 *   the rest       as chunk_meta_build; the checks run on the int64 values.
 *
 * One kernel launch; no host synchronisation; graph-capturable.  Host errors as
 * chunk_meta_build, plus INVALID_ARG for a NULL cu_seqlens32.
 */
gcl_status_t chunk_meta_build_i64(const int64_t *cu_seqlens, int32_t n_max, int64_t t_max,
                                  int32_t bt, int64_t nt_max, int32_t *cu_seqlens32,
                                  int32_t *chunk_indices, int32_t *chunk_offsets, int32_t *seq_order,
                                  int32_t *dev_status, gcl_stream_t stream);

/*
 * Forward arguments (GDN and KDA).  All pointers are device pointers.
 */
typedef struct gcl_fwd_args {
    const void *q;                 /* [t_max, H, K]  dtype                                   */
    const void *k;                 /* [t_max, H, K]  dtype                                   */
    const void *v;                 /* [t_max, H, V]  dtype                                   */
    const float *g;                /* GDN [t_max, H]; KDA [t_max, H, K]; fp32 log gate <= 0  */
    const void *beta;              /* [t_max, H]  dtype                                      */
    const float *h0;               /* [n_max, H, K, V] fp32, or NULL for a zero state        */
    const int32_t *cu_seqlens;     /* [n_max + 1] int32                                      */
    const int32_t *chunk_indices;  /* [nt_max, 2] from chunk_meta_build (tensor-core path)   */
    const int32_t *chunk_offsets;  /* [n_max + 1] from chunk_meta_build                      */
    const int32_t *seq_order;      /* [n_max] from chunk_meta_build, or NULL (index order)   */
    void *o;                       /* [t_max, H, V] dtype (out); live rows only; may be NULL */
    float *ht;                     /* [n_max, H, K, V] fp32 (out) or NULL                    */
    float *h_save;                 /* [nt_max, H, K, V] fp32 (out) or NULL: the state before */
                                   /* chunk i of sequence n at row chunk_offsets[n] + i      */
    int32_t *dev_status;           /* [1] or NULL: no work if non-zero on entry; set to      */
                                   /* GCL_DEV_BAD_RANGE if a sequence range is invalid       */
    void *workspace;               /* device scratch, at least                               */
    size_t workspace_bytes;        /* gcl_fwd_workspace_min_bytes() bytes                    */
    int64_t t_max;                 /* token capacity of every [t_max, ...] buffer            */
    int32_t n_max;                 /* sequence capacity (cu_seqlens has n_max + 1 entries)   */
    int32_t H, K, V;               /* heads, key dim, value dim                              */
    int32_t bt;                    /* chunk size: 64, or 32 (CUDA-core kernel only)          */
    float scale;                   /* read-out scale, usually K^-1/2                         */
    int32_t dtype;                 /* gcl_dtype_t of q, k, v, beta, o                        */
} gcl_fwd_args;

/* Bytes of device workspace the forward's fastest launch plan uses for these sizes, and
 * the least it accepts.
 *
 * Sizes the CUDA cores serve (fp32 inputs, K or V = 64, bt = 32, and the KDA forward
 * with fp16 inputs) have two plans: one fp32 kernel, which needs no workspace (the
 * minimum, 0), and the split plan, fastest, whose records are per chunk row and head the
 * fp32 matrices W, Q', K' [BT x K], L [BT x BT] (rows padded by 4 floats), Gamma_c [K]
 * and U [BT x V] (84.25 KiB at K = V = 64, BT = 64; 148.5 KiB at K = V = 128), for K = V
 * only; it runs whenever the workspace holds them and chunk_indices and chunk_offsets are
 * given.
 *
 * The tensor-core path has two plans.  The W form keeps per chunk and head the
 * inverted intra-chunk matrix T and the masked decayed QK^T, 25 KiB (bf16); it is
 * the minimum.  The transition form keeps per chunk and head the chunk's affine
 * state map and output map (N, B, Y, Z below, bf16), 96 KiB; it shortens the serial
 * step per chunk and is the fastest plan when each head is split over 4 or more
 * value-column slices (few sequence-head units).  A forward that writes h_save
 * (training) also takes the transition form, because its records are what the
 * backward's state-gradient sweep reads (gcl_bwd_args.fwd_workspace).  The forward
 * runs that plan whenever its scratch fits in workspace_bytes, else the W form, so any
 * workspace of at least the minimum works; given sizes always select the same plan. */
size_t gcl_fwd_workspace_bytes(const gcl_fwd_args *args);
size_t gcl_fwd_workspace_min_bytes(const gcl_fwd_args *args);
/* With at least as many sequence-head units as SMs (n_max * H >= the device's SM count) a
 * GDN forward runs the fused plan,
 * which needs no workspace: without h_save both queries return 0 and workspace may be
 * NULL; with h_save (a training forward) the fastest plan stays the transition form
 * (its records serve the backward) and the fused plan runs with any smaller workspace. */

/* Bytes of device workspace kda_chunk_fwd's fastest plan needs for these sizes (on the
 * CUDA cores: the split plan's records, as above).  KDA on the tensor cores runs the
 * transition form (96.5 KiB per chunk and head: the chunk's affine state map and
 * output map, and the per-key-channel state decay of the chunk); a workspace
 * smaller than those records returns GCL_ERR_CAPACITY.  When the fastest plan is
 * segmented (gcl_fwd_chain_segments) it also holds the segment buffers; without
 * room for them the forward runs the plain chain.  gcl_fwd_workspace_bytes and
 * gcl_fwd_workspace_min_bytes describe gdn_chunk_fwd only. */
size_t gcl_kda_fwd_workspace_bytes(const gcl_fwd_args *args);

/*
 * Segments per sequence of the fastest tensor-core forward plan (GDN and KDA, bf16,
 * K = V = 128, workspace of the fastest size) for these capacities; 0 when every
 * (sequence, head, column slice) runs its whole chain in one CTA.
 *
 * With few sequence-head units (n_max * H at most SMs / 24) and long sequences
 * (NT_max at least 4 P n_max chunks), the forward cuts each sequence of nc chunks into
 * P segments of ceil(nc / P) chunks, following HA-NPU section 4 (third tier: a
 * long head's chunks spread over cores) and the Map-Reduce-Map split of its
 * section 2.1, with the transition form's affine chunk maps as the unit of work.
 * After the chunk records come three launches:
 *   summaries  each segment but the last: its affine map S_end = M S_start + B over its
 *              chunks, from the state [I | 0] over 256 columns;
 *   scan       the start states S(s + 1) = M(s) S(s) + B(s) from S(0) = h0, in fp32;
 *   outputs    each segment's recurrence from its start state (o, h_save), ht from
 *              the last segment.
 * Segment buffers: n_max * H * P * 192 KiB after the records.  The result depends
 * only on the capacities and the device's SM count, so a captured graph keeps its
 * plan.  Returns 0 for invalid sizes.
 */
int32_t gcl_fwd_chain_segments(int64_t t_max, int32_t n_max, int32_t H, int32_t bt);

/*
 * The launch plan a forward with these arguments runs (workspace_bytes included), for
 * callers that size graphs or count launches, and for tests:
 *   GCL_PLAN_CUDA_CORES  one fp32 CUDA-core kernel (fp32 inputs, K or V = 64, bt = 32, fp16 KDA)
 *   GCL_PLAN_CUDA_CORES_SPLIT  the same sizes (K = V) as a chunk prep over every chunk and head
 *                        plus a chain over value-column slices (HA-NPU section 2.1: only the
 *                        Reduce is serial), when the workspace holds the prep's records
 *   GCL_PLAN_FUSED       one tensor-core kernel per (sequence, head), everything on chip
 *                        (GDN, n_max * H >= SMs: HA-NPU section 4, first tier)
 *   GCL_PLAN_W_FORM      chunk prep (T, L records) + chain over value-column slices
 *   GCL_PLAN_TRANSITION  chunk prep (affine chunk maps) + chain over value-column slices
 *   GCL_PLAN_SEGMENTED   the transition plan with the segment-parallel chain
 * Every plan but the segmented one runs chunk_meta_build's output through one or two
 * launches; the segmented plan adds the segment summaries, the scan and the segment outputs.  Returns -1
 * for arguments the forward would reject on the host.  gcl_fwd_plan describes
 * gdn_chunk_fwd, gcl_kda_fwd_plan kda_chunk_fwd.
 */
typedef enum {
    GCL_PLAN_CUDA_CORES = 0,
    GCL_PLAN_FUSED = 1,
    GCL_PLAN_W_FORM = 2,
    GCL_PLAN_TRANSITION = 3,
    GCL_PLAN_SEGMENTED = 4,
    GCL_PLAN_CUDA_CORES_SPLIT = 5
} gcl_fwd_plan_t;
int32_t gcl_fwd_plan(const gcl_fwd_args *args);
int32_t gcl_kda_fwd_plan(const gcl_fwd_args *args);

/*
 * gdn_chunk_fwd -- gated delta rule prefill: o and ht from q, k, v, g, beta, h0.
 * kda_chunk_fwd -- the same with the per-key-channel gate of KDA.
 *
 * Each (sequence, head) runs the chunkwise Map-Reduce-Map pipeline (HA-NPU
 * sections 2.1 and 4; FLA RFC "Step 3": gate/chunk cumsum -> intra (KK^T and
 * triangular solve) -> recompute_w_u -> h -> o) in one fused launch with the
 * state held on chip; the value dimension of each head may be split across
 * CTAs (HA-NPU section 4, column-wise split without cross-core reductions).
 * Zero-length sequences write ht = h0 (or zeros).
 *
 * Supported: bt in {32, 64} (the RFC's test matrix, "BT=32 and BT=64"); K, V in
 * {64, 128}; dtype GCL_F32, GCL_BF16 or GCL_F16.  GDN and KDA with bf16 inputs,
 * and GDN with fp16 inputs (the fused and transition plans, every MMA operand and record
 * in fp16), K = V = 128 and bt = 64 run on the tensor cores (tcgen05).  With many sequence-head
 * units a GDN forward runs the fused plan: one CTA per (sequence, head)
 * walks its chunks with every intermediate (the gate cumsum, A, T = (I + A)^-1, L, the
 * GEMM-first R = diag(beta)(V - diag(Gamma) K S), E = T R, the state) on chip, so only
 * the inputs are read and o, ht written (HA-NPU sections 4 and 5).  Otherwise a
 * chunk-parallel launch over chunk_indices forms per chunk either T = (I + A)^-1
 * and L (W form, GDN) or the chunk's transition S' = Gamma_c S + N S + B and
 * output O = Y S + Z (transition form; for KDA Gamma_c is a per-key-channel
 * diagonal) into the workspace, then the per-(sequence, head, column slice)
 * launch runs the state recurrence.  Everything else runs the fp32 CUDA-core
 * kernel.  The workspace of kda_chunk_fwd is sized by gcl_kda_fwd_workspace_bytes.
 * Pointers must be 16-byte aligned.
 */
gcl_status_t gdn_chunk_fwd(const gcl_fwd_args *args, gcl_stream_t stream);
gcl_status_t kda_chunk_fwd(const gcl_fwd_args *args, gcl_stream_t stream);

/*
 * gdn_chunk_fwd_noalloc -- gdn_chunk_fwd for callers that cannot allocate device
 * memory.  The paper has no counterpart; this is a convenience of this library.
 *
 * Some callers cannot hand the forward a workspace: code running inside a CUDA
 * graph capture whose allocator is not capture-aware, runtimes that fix their
 * memory budget at start-up and forbid later cudaMalloc calls, and plugin hosts
 * that pass tensors in but offer no allocator.  This entry point takes the same
 * arguments as gdn_chunk_fwd but ignores args->workspace / workspace_bytes: the
 * scratch lives in a static device array of gcl_noalloc_scratch_bytes() bytes
 * (32 MiB) inside the library, which every GPU that loads the library holds
 * until the process exits.  It allocates and frees nothing.
 *
 *  - Sizes whose minimum scratch (gcl_fwd_workspace_min_bytes) exceeds that limit
 *    return GCL_ERR_CAPACITY before any work is enqueued.  The bf16 K = V = 128
 *    path needs at least 25 KiB per chunk and head, i.e. up to 1310 chunk-heads
 *    (for example T = 4096 tokens with 16 heads).  The plan is the fastest one
 *    whose scratch fits in the array.
 *  - The first call on a device looks up the array's device address (with that
 *    device current) and caches it; make that first call before any stream
 *    capture.
 *  - All calls on a device share the array and leave their contents in it;
 *    calls whose GPU executions overlap (unordered streams, concurrent graph
 *    replays) race on it and give wrong results.
 */
gcl_status_t gdn_chunk_fwd_noalloc(const gcl_fwd_args *args, gcl_stream_t stream);

/* Size in bytes of the static scratch array used by gdn_chunk_fwd_noalloc. */
size_t gcl_noalloc_scratch_bytes(void);

/*
 * gcl_selftest_wait_timeout -- a self-test of the bounded waits.  Every mbarrier
 * wait of the tensor-core kernels gives up after a time limit (0.2 s), records
 * GCL_DEV_WAIT_TIMEOUT in the device status word and returns, so that a lost copy
 * or MMA completion becomes a status the host can read rather than a hung GPU.  This
 * call launches one CTA that waits on an mbarrier nothing arrives at: after the
 * limit *dev_status holds GCL_DEV_WAIT_TIMEOUT (if it was 0) and the context stays
 * usable.  No fault, trap or hang.  Host error: INVALID_ARG for a NULL dev_status.
 */
gcl_status_t gcl_selftest_wait_timeout(int32_t *dev_status, gcl_stream_t stream);

/*
 * Backward arguments (GDN and KDA).  All pointers are device pointers.
 */
typedef struct gcl_bwd_args {
    const void *q, *k, *v;         /* as in gcl_fwd_args                                     */
    const float *g;                /* GDN [t_max, H]; KDA [t_max, H, K]; fp32                */
    const void *beta;              /* [t_max, H] dtype                                       */
    const float *h0;               /* [n_max, H, K, V] or NULL                               */
    const void *d_o;               /* [t_max, H, V] dtype: gradient of the loss w.r.t. o     */
    const float *dht;              /* [n_max, H, K, V] fp32 or NULL: gradient w.r.t. ht      */
    const int32_t *cu_seqlens;     /* [n_max + 1]                                            */
    const int32_t *chunk_indices;  /* [nt_max, 2] from chunk_meta_build                      */
    const int32_t *chunk_offsets;  /* [n_max + 1] from chunk_meta_build                      */
    const float *h_save;           /* [nt_max, H, K, V] from the forward, or NULL: then the  */
                                   /* states are recomputed into the workspace              */
    float *dq, *dk;                /* [t_max, H, K] fp32 (out), live rows                    */
    float *dv;                     /* [t_max, H, V] fp32 (out)                               */
    float *dg;                     /* shape of g, fp32 (out): w.r.t. the raw log gate g      */
    float *dbeta;                  /* [t_max, H] fp32 (out)                                  */
    float *dh0;                    /* [n_max, H, K, V] fp32 (out) or NULL                    */
    void *workspace;               /* device scratch of gcl_bwd_workspace_bytes() bytes      */
    size_t workspace_bytes;
    int32_t *dev_status;           /* as in gcl_fwd_args                                     */
    int64_t t_max;
    int32_t n_max, H, K, V, bt;
    float scale;
    int32_t dtype;
    const void *fwd_workspace;     /* the workspace of the forward call that wrote h_save,   */
    size_t fwd_workspace_bytes;    /* or NULL: its chunk records are then reused (below)     */
} gcl_bwd_args;

/* Bytes of device workspace gdn_chunk_bwd (gcl_bwd_workspace_bytes) and
 * kda_chunk_bwd (gcl_kda_bwd_workspace_bytes) need for these sizes (depends on
 * whether h_save and fwd_workspace are NULL).  Returns 0 for unsupported sizes.
 *
 * Chunk records.  On the tensor cores (bf16, K = V = 128, bt = 64) the reverse
 * state-gradient sweep reads each chunk's transition-form records (the affine state
 * map N, B of the chunk; see gdn_chunk_fwd).  A forward that writes h_save (a
 * training forward) runs the transition plan whenever its workspace holds it, so
 * its workspace then holds exactly these records: pass that workspace and its size as
 * fwd_workspace / fwd_workspace_bytes, with the same inputs and h_save, and the
 * backward reads them instead of recomputing them (the caller guarantees that the
 * forward ran on these inputs, as for h_save).  The backward decides from the sizes
 * alone whether that forward ran the transition plan and ignores fwd_workspace
 * otherwise.  Without h_save the backward's own recompute of the states runs the
 * transition plan and reuses its records. */
size_t gcl_bwd_workspace_bytes(const gcl_bwd_args *args);
size_t gcl_kda_bwd_workspace_bytes(const gcl_bwd_args *args);

/*
 * gdn_chunk_bwd -- gradients dq, dk, dv, dg, dbeta, dh0 of
 *   L(o, ht) with upstream gradients d_o and dht,
 * through the GDN chunk forward (FLA RFC "Step 3": recomputation, state, WY,
 * gate and gradient kernels).  A reverse sweep over the chunks of each
 * (sequence, head) carries the state gradient; the per-chunk gradients are then
 * computed in parallel over chunk_indices, whose sentinel rows exit at once.
 * Supported sizes as for the forward.  bf16 with K = V = 128 runs on the tensor
 * cores (tcgen05), everything else on the CUDA cores in fp32.
 *
 * kda_chunk_bwd -- the same through the KDA chunk forward (per-key-channel gate;
 * dg has the shape of g, [t_max, H, K]).  For bf16 with K = V = 128 the reverse
 * state-gradient sweep runs on the tensor cores (tcgen05, from the KDA transition
 * records: the forward's when handed over, else recomputed) and the chunk gradients
 * on the CUDA cores in fp32; every other size and dtype runs both on the CUDA cores in
 * fp32.  The recompute of missing states uses the forward's own path.  Errors as for
 * gdn_chunk_bwd.
 */
gcl_status_t gdn_chunk_bwd(const gcl_bwd_args *args, gcl_stream_t stream);
gcl_status_t kda_chunk_bwd(const gcl_bwd_args *args, gcl_stream_t stream);

/*
 * causal_conv1d -- the short causal depthwise convolution that precedes the chunk
 * attention in the layer (FLA RFC "[RFC] Add Graph Capture Support for FLA Prefill and
 * Training Paths on Ascend NPUs", section "Step 3": dense and varlen inputs, forward and
 * backward, bias, activation and residual paths, initial and final states, fixed chunk
 * metadata and state buffers; section "API proposal": the same chunk_indices as the chunk
 * attention).  The pages print no formula; this library computes, per channel d and for
 * the inputs xx_n(i) of sequence n (xx_n(i) = x[bos_n + i] for i >= 0, h0[n, d, W - 1 + i]
 * for -(W - 1) <= i < 0, zeros without h0):
 *
 *   y[bos_n + p, d] = act(bias[d] + sum_{j<W} weight[d, j] xx_n(p - (W - 1) + j)) + residual
 *   ht[n, d, k] = xx_n(len_n - (W - 1) + k),   k = 0 .. W - 2 (oldest first)
 *
 * act is the identity or SiLU (z / (1 + exp(-z))).  Zero-length sequences write ht = h0.
 * The backward returns dx, dweight, dbias, dh0 of <dy, y> + <dht, ht> (the gradient of the
 * residual is dy itself).  One struct serves both directions; fields of the other direction
 * are ignored.  All pointers are device pointers.
 *
 * Supported: W in {2, 3, 4}; D a multiple of 8; bt = 64; dtype GCL_F32 or GCL_BF16 for x,
 * weight, bias, residual, h0, y, ht and dy (the gradients are fp32); x, y, residual, dy and
 * dx 16-byte aligned.  Launch shapes depend only on (nt_max, n_max, D); every call is
 * graph-capturable.  Errors: INVALID_ARG / UNSUPPORTED on the host before anything is
 * enqueued, data errors through dev_status as for the chunk attention.
 */
typedef enum { GCL_ACT_NONE = 0, GCL_ACT_SILU = 1 } gcl_activation_t;

typedef struct gcl_conv_args {
    const void *x;                 /* [t_max, D] dtype                                       */
    const void *weight;            /* [D, W] dtype                                           */
    const void *bias;              /* [D] dtype or NULL                                      */
    const void *residual;          /* [t_max, D] dtype or NULL: added after the activation   */
    const void *h0;                /* [n_max, D, W - 1] dtype or NULL (zeros)                */
    void *y;                       /* forward: [t_max, D] dtype (out), live rows only        */
    void *ht;                      /* forward: [n_max, D, W - 1] dtype (out) or NULL         */
    const void *dy;                /* backward: [t_max, D] dtype, the gradient w.r.t. y      */
    const float *dht;              /* backward: [n_max, D, W - 1] fp32 or NULL               */
    float *dx;                     /* backward: [t_max, D] fp32 (out), live rows only        */
    float *dweight;                /* backward: [D, W] fp32 (out)                            */
    float *dbias;                  /* backward: [D] fp32 (out) or NULL                       */
    float *dh0;                    /* backward: [n_max, D, W - 1] fp32 (out) or NULL         */
    const int32_t *cu_seqlens;     /* [n_max + 1] int32                                      */
    const int32_t *chunk_indices;  /* [nt_max, 2] from chunk_meta_build (bt = 64)            */
    int32_t *dev_status;           /* [1] or NULL, as in gcl_fwd_args                        */
    void *workspace;               /* backward: gcl_causal_conv1d_bwd_workspace_bytes()      */
    size_t workspace_bytes;        /*   bytes (per-chunk partial sums of dweight, dbias)     */
    int64_t t_max;                 /* token capacity                                         */
    int32_t n_max, D, W, bt;       /* sequences, channels, taps, chunk size                  */
    int32_t activation;            /* gcl_activation_t                                       */
    int32_t dtype;                 /* gcl_dtype_t                                            */
} gcl_conv_args;

gcl_status_t causal_conv1d_fwd(const gcl_conv_args *args, gcl_stream_t stream);
size_t gcl_causal_conv1d_bwd_workspace_bytes(const gcl_conv_args *args);
gcl_status_t causal_conv1d_bwd(const gcl_conv_args *args, gcl_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GCL_H */
