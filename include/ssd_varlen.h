/*
 * ssd_varlen.h -- C ABI of the GB300 Mamba2 SSD varlen prefill library.
 *
 * The operation (one layer, one call):
 *   Tokens of R requests are packed as x (T,H,P) with cu_seqlens (R+1) marking
 *   where each request starts; there is no padding and no batch dimension
 *   ("[Model] Mamba2 varlen and metadata refactor", Purpose item 1).  For every
 *   request i and head h, with group g = h / (H/G), the SSD scan runs
 *       dt'  = softplus(dt[t,h] + dt_bias[h])
 *       h_t  = exp(dt' A[h]) h_{t-1} + dt' x[t,h,:] (outer) B[t,g,:]     (P x N)
 *       y[t,h,:] = (h_t C[t,g,:] + D[h] x[t,h,:]) * silu(z[t,h,:])
 *   starting from the request's initial state (a pool slot, or zeros), which
 *   must decay from the request's first token even inside a partial first
 *   chunk ("[Bugfix] Mamba2 SSD varlen bug fix initstates decay, improve test,
 *   assert chunk pwr 2", instinctive explanation items 1-4).  chunk_size is a
 *   power of two and does not change the result (same page, Purpose note).
 *   Optional state outputs: the final state per request (dense and/or into a
 *   pool slot), the state after every chunk (per-chunk intermediate-state
 *   export), and the state at every block boundary scattered into pool slots
 *   through a per-request block table ("Automatic prefix caching for GDN hybrid
 *   models (mamba_cache_mode=all) with MTP speculative decoding", Purpose and
 *   Kernels/layers: intermediate-state export, block-aligned checkpoint
 *   scatter, dual read/write state anchors).
 *
 * Chunks are cut at ABSOLUTE positions: a request with s = num_computed[i]
 * tokens already in its state covers positions [s, s+L_i); chunk boundaries are
 * the multiples of chunk_size, block boundaries the multiples of block_size.
 * Chunk j of request i is row chunk_first[i] + j of the export buffer, where
 * chunk_first is the exclusive prefix sum of the per-request chunk counts; its
 * exported state is the state after the chunk's last token.  A block boundary
 * kb (s < kb <= s+L_i) writes the state after position kb-1 to
 * state_pool[block_table[i*block_table_width + kb/block_size - 1]]; entries < 0
 * are skipped.
 *
 * Layouts: row-major, last index fastest.  x, z, y (T,H,P); B, C (T,G,N);
 * dt (T,H); dt_bias, A, D (H) fp32; states (..., H, P, N) fp32.
 * x, dt, B, C, z, y share one dtype (bf16 or fp32).
 *
 * Ownership: the caller allocates every buffer, device workspace included;
 * the library allocates nothing and launches only on the stream it is given.
 * Every device pointer must be 16-byte aligned and every tensor contiguous.
 *
 * Errors: host-detectable problems return a negative ssd_status and launch
 * nothing.  Problems only the device can see (a cu_seqlens entry out of
 * order, a slot or table entry out of range) set bits in a device error word
 * held in the workspace; the offending read is treated as zeros and the
 * offending write is skipped.  Nothing traps.  ssd_varlen_status reads and
 * clears the word (it synchronises the plan's stream).
 */
#ifndef SSD_VARLEN_H
#define SSD_VARLEN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum ssd_dtype { SSD_DTYPE_BF16 = 0, SSD_DTYPE_F32 = 1 };

enum ssd_status {
    SSD_OK = 0,
    SSD_ERR_NULL = -1,          /* a required pointer is NULL */
    SSD_ERR_DIMS = -2,          /* a size is out of range (T, R, H, P, N, G, slots) */
    SSD_ERR_CHUNK_SIZE = -3,    /* chunk_size is not an integer power of 2 in [16, 256] */
    SSD_ERR_GROUPS = -4,        /* H is not a multiple of G */
    SSD_ERR_BLOCK_SIZE = -5,    /* block_size is not a multiple of chunk_size */
    SSD_ERR_DTYPE = -6,         /* unknown dtype */
    SSD_ERR_ALIGN = -7,         /* a device pointer is not 16-byte aligned */
    SSD_ERR_WORKSPACE = -8,     /* workspace too small or misaligned */
    SSD_ERR_PLAN = -9,          /* plan not built, or built for other dims */
    SSD_ERR_CUDA = -10,         /* a CUDA runtime call failed */
    SSD_ERR_UNSUPPORTED = -11   /* a combination this library does not handle */
};

/* Bits of the device error word (ssd_varlen_status). */
#define SSD_DEVERR_CU_SEQLENS 0x1    /* cu_seqlens[0] != 0, decreasing, or cu[R] != T */
#define SSD_DEVERR_NUM_COMPUTED 0x2  /* negative num_computed, or s + L beyond 2^31 - 1 */
#define SSD_DEVERR_INIT_SLOT 0x4     /* init slot >= num_slots (read as zeros) */
#define SSD_DEVERR_FINAL_SLOT 0x8    /* final slot >= num_slots (write skipped) */
#define SSD_DEVERR_BLOCK_SLOT 0x10   /* block-table slot >= num_slots (write skipped) */
#define SSD_DEVERR_BLOCK_TABLE 0x20  /* a boundary needs a column >= block_table_width */
#define SSD_DEVERR_TIMEOUT 0x40      /* a bounded wait inside a kernel gave up (work skipped) */
#define SSD_DEVERR_INTERNAL 0x80     /* a kernel could not start (shared-memory alignment) */
#define SSD_DEVERR_ALIAS 0x100       /* ssd_varlen_check_slots: a written slot is read or written twice */

/* Problem sizes.  Filled by the caller, copied into the plan. */
typedef struct ssd_dims {
    int64_t T;                 /* total tokens, >= 0 */
    int32_t R;                 /* requests, >= 1 */
    int32_t H, P, N, G;        /* heads, headdim, d_state, groups (H % G == 0) */
    int32_t chunk_size;        /* power of 2 in [16, 256] */
    int32_t dtype;             /* enum ssd_dtype of x, dt, B, C, z, y */
    int32_t num_slots;         /* rows of state_pool (0 when no pool is used) */
    int32_t block_size;        /* block-checkpoint granularity; 0 = no scatter */
    int32_t block_table_width; /* columns of block_table */
    int32_t reserved;          /* must be 0 */
} ssd_dims;

/* Per-batch plan: host-side handle to device metadata kept in the workspace.
 * Built once per batch by ssd_varlen_plan and reused by every layer's
 * ssd_varlen_forward while cu_seqlens / num_computed stay unchanged.  The
 * fields are the library's; callers treat the struct as opaque. */
typedef struct ssd_plan {
    ssd_dims dims;
    void *workspace;
    size_t workspace_bytes;
    const int32_t *cu_seqlens;
    const int32_t *num_computed;
    int64_t max_chunks;        /* bound on export rows: ceil(T/Q) + R */
    int64_t max_segs;          /* bound on work segments */
    int32_t seg_len;           /* tokens per work segment (multiple of 128) */
    int32_t flags;
    uint64_t magic;
    cudaStream_t stream;       /* the stream the plan was built on */
} ssd_plan;

/* Inputs and outputs of a forward.  With T = 0 (every request empty) the token
 * buffers (x, dt, B, C, z, y) may be NULL; the forward then writes each
 * request's final state (its initial state, or zeros) where asked. */
typedef struct ssd_inputs {
    const void *x;             /* (T,H,P) */
    const void *dt;            /* (T,H) */
    const float *dt_bias;      /* (H) */
    const float *A;            /* (H) */
    const void *B;             /* (T,G,N) */
    const void *C;             /* (T,G,N) */
    const float *D;            /* (H) or NULL: no skip term */
    const void *z;             /* (T,H,P) or NULL: no gate */
    const int32_t *init_slots; /* (R) or NULL: every request starts from zeros; -1 = zeros */
    float *state_pool;         /* (num_slots,H,P,N) or NULL; read through init_slots,
                                  written through final_slots and block_table */
} ssd_inputs;

typedef struct ssd_outputs {
    void *y;                   /* (T,H,P), required */
    float *final_states;       /* (R,H,P,N) or NULL */
    const int32_t *final_slots;/* (R) or NULL; -1 = do not write that request */
    float *chunk_states;       /* (n_chunks,H,P,N) or NULL; n_chunks = ssd_varlen_count_chunks */
    const int32_t *block_table;/* (R, block_table_width) or NULL; needs block_size > 0 */
} ssd_outputs;

/* Bytes of device workspace the plan and forward need for these dims. */
size_t ssd_varlen_workspace_size(const ssd_dims *dims);

/* Export rows for a batch, from HOST copies of cu_seqlens (R+1) and
 * num_computed (R, or NULL for zeros).  Negative on bad input. */
int64_t ssd_varlen_count_chunks(const int32_t *cu_seqlens_host, const int32_t *num_computed_host,
                                int32_t R, int32_t chunk_size);

/* Validates dims, then launches the device metadata builder on `stream`:
 * per-request chunk and segment offsets and the segment work list, computed
 * from cu_seqlens (device, R+1) and num_computed (device, R, or NULL) without
 * a host synchronisation.  Fills *out.  The workspace (16-byte aligned, at
 * least ssd_varlen_workspace_size bytes) holds the metadata until the next
 * plan on it. */
int ssd_varlen_plan(const ssd_dims *dims, const int32_t *cu_seqlens, const int32_t *num_computed,
                    void *workspace, size_t workspace_bytes, cudaStream_t stream, ssd_plan *out);

/* One SSD varlen prefill over the planned batch, launched on `stream`
 * (normally the plan's stream; another stream must be ordered after it).
 * Writes y and whichever state outputs are non-NULL.  Write slots must not
 * alias slots read in the same call.
 *
 * Its kernels are programmatic dependent launches: each may become resident
 * before the stream's previous kernel has finished, but waits
 * (griddepcontrol.wait) for it, and for its writes to be visible, before
 * touching global memory, so stream order holds as for plain launches.  The
 * plan's kernel is launched the same way, and lets the next kernel on its
 * stream be scheduled at its start; a caller kernel launched there with the
 * same attribute must wait likewise.
 * Both calls can be captured into a CUDA graph. */
int ssd_varlen_forward(const ssd_plan *plan, const ssd_inputs *in, const ssd_outputs *out,
                       cudaStream_t stream);

/* Synchronises the plan's stream (only that stream), returns the device error
 * bits in *device_err and clears them.  Returns SSD_OK or SSD_ERR_CUDA. */
int ssd_varlen_status(const ssd_plan *plan, int *device_err);

/* Which kernel path ssd_varlen_forward takes for these arguments, without
 * launching anything (same validation and return codes as the forward).
 *   SSD_PATH_TENSOR_CORE_PAIRED: the fused chunked scan on the tensor cores
 *     (tcgen05, TMEM, TMA) with two heads of a group per CTA sharing their B
 *     and C tiles: bf16, P = 64, N = 128 and an even number of heads per group.
 *   SSD_PATH_TENSOR_CORE: the same scan with one head per CTA: the other bf16
 *     shapes with P in {64, 128} and N = 128.
 *   For both, *tile (nullable) receives the internal tile length in tokens:
 *     128, or the chunk / block granularity when exports or block checkpoints
 *     need a finer cut.  The result does not depend on the tile (chunk_size
 *     only decides where exports fall: "[Bugfix] Mamba2 SSD varlen bug fix
 *     initstates decay", Purpose).
 *   SSD_PATH_GENERAL: a token-serial recurrence on the CUDA cores, for fp32
 *     inputs, every other bf16 shape and an all-empty batch; correct but one to
 *     two orders of magnitude slower per token than the tensor-core path.
 *     *tile receives 1. */
enum ssd_path { SSD_PATH_TENSOR_CORE = 1, SSD_PATH_GENERAL = 2, SSD_PATH_TENSOR_CORE_PAIRED = 3 };
int ssd_varlen_forward_path(const ssd_plan *plan, const ssd_inputs *in, const ssd_outputs *out, int *path,
                            int *tile);

/* Static description of a status code or device error bit set. */
const char *ssd_varlen_strerror(int code);

/* ---- Forward without a caller-provided workspace -------------------------
 * Not described by the pages (there is no counterpart there): it exists for
 * callers that cannot allocate device memory for a workspace -- a plugin
 * running inside a serving process or framework that owns the device memory
 * pool, or a latency-critical loop where cudaMalloc (which can synchronise the
 * device and can fail under memory pressure) is not allowed.
 *
 * Runs the same metadata builder and forward as ssd_varlen_plan +
 * ssd_varlen_forward, with the workspace taken from a fixed array in device
 * memory that the library owns: SSD_STATIC_SCRATCH_BYTES bytes, held on each
 * GPU that loads the library until the process exits.  The function itself
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library call);
 * the caller still allocates every input and output buffer.
 *
 * - Problems whose workspace (ssd_varlen_workspace_size) exceeds
 *   SSD_STATIC_SCRATCH_BYTES are rejected with SSD_ERR_WORKSPACE before any
 *   launch; invalid dims return the same codes as ssd_varlen_plan.
 * - The first call on a device looks up the array's device address with that
 *   device current (cudaGetSymbolAddress); make that first call before any
 *   stream capture on the device.  The address is kept for the life of the
 *   process: do not call this entry point again on a device after
 *   cudaDeviceReset on it (the array may then live elsewhere).
 * - Every call shares the one array, which keeps the previous call's
 *   contents.  Calls whose GPU work overlaps (different streams or host
 *   threads without ordering) race on it: order them on one stream.  Each
 *   call's metadata builder rewrites the error word and counters first.
 * - plan_out (nullable) receives the plan of this call, valid until the next
 *   call; pass it to ssd_varlen_status to read this call's device errors.
 */
#define SSD_STATIC_SCRATCH_BYTES (32u << 20)
int ssd_varlen_forward_static(const ssd_dims *dims, const int32_t *cu_seqlens, const int32_t *num_computed,
                              const ssd_inputs *in, const ssd_outputs *out, cudaStream_t stream,
                              ssd_plan *plan_out);

/* ---- Decode and speculative-decode step with dual read/write anchors -----
 * "Automatic prefix caching for GDN hybrid models (mamba_cache_mode=all) with
 * MTP speculative decoding", Purpose (the Kernels/layers bullet): the decode
 * kernels take dual read/write state anchors, so that a speculative-decode step
 * reads the previous step's running state from one slot while writing the
 * current step's states to others.  The same recurrence as the forward above,
 * for short per-request windows:
 *
 *   Request i owns tokens [cu_seqlens[i], cu_seqlens[i+1]) of the packed batch:
 *   one token for a plain decode step, 1 + the number of draft tokens for a
 *   speculative step (0 tokens: nothing is read or written for it).  For every
 *   head h its state starts from state_pool[read_slots[i]] (the read anchor;
 *   read_slots[i] < 0 starts from zeros) and advances token by token; y of each
 *   token is written, and the state after token t goes to
 *   state_pool[write_slots[t]] when write_slots[t] >= 0 (the write anchors:
 *   the state after every draft position can be kept, so the step after
 *   verification reads the one after the last accepted token).
 *
 * dims: T, R, H, P, N, G, dtype, num_slots (>= 1) as above; chunk_size,
 * block_size and block_table_width are not used.  P * N must be at most 16384
 * and N a power of two in [16, 256] (SSD_ERR_UNSUPPORTED otherwise).  A write
 * slot must not be a slot read in the same call.  Layouts as above; write_slots
 * is (T) int32 and nullable (no state written), z and D are nullable.
 * device_err (one int32 in device memory, required) receives SSD_DEVERR_* bits
 * (CU_SEQLENS, INIT_SLOT for a read slot >= num_slots, FINAL_SLOT for a write
 * slot >= num_slots); the caller clears it.  With T = 0 the token buffers (x,
 * dt, B, C, z, y) may be NULL.  Launches one kernel on `stream`; allocates
 * nothing. */
typedef struct ssd_decode_io {
    const void *x, *dt;         /* (T,H,P), (T,H) in dims.dtype */
    const float *dt_bias, *A;   /* (H) */
    const void *B, *C;          /* (T,G,N) in dims.dtype */
    const float *D;             /* (H) or NULL */
    const void *z;              /* (T,H,P) or NULL */
    float *state_pool;          /* (num_slots,H,P,N) fp32, read and written */
    const int32_t *read_slots;  /* (R) read anchor per request, < 0 = zero state */
    const int32_t *write_slots; /* (T) write anchor per token, < 0 = none; or NULL */
    void *y;                    /* (T,H,P) in dims.dtype */
    int32_t *device_err;        /* one int32, OR-ed with SSD_DEVERR_* bits */
} ssd_decode_io;

int ssd_varlen_decode(const ssd_dims *dims, const int32_t *cu_seqlens, const ssd_decode_io *io,
                      cudaStream_t stream);

/* ---- Varlen causal depthwise conv1d with conv-state anchors ---------------
 * The step before the SSD in a Mamba2 layer, over the same packed varlen batch
 * ("[Model] Mamba2 varlen and metadata refactor", Purpose items 1-2; the
 * causal_conv1d decode kernel with dual read/write state anchors of "Automatic
 * prefix caching for GDN hybrid models (mamba_cache_mode=all) with MTP
 * speculative decoding", Purpose, Kernels/layers).  Per request i (tokens
 * [cu_seqlens[i], cu_seqlens[i+1])) and channel c, with the request's inputs
 * preceded by its W-1 conv-state values (oldest first):
 *     y[t,c] = act(bias[c] + sum_{k<W} weight[c,k] * xin[t - (W-1) + k, c])
 * the conv state read from conv_pool[read_slots[i]] (zeros when the slot is < 0
 * or read_slots is NULL) and the last W-1 inputs (the initial values included
 * when the request is shorter) written to conv_pool[write_slots[i]] when that
 * slot is >= 0; act is SiLU when dims.silu != 0, else the identity.
 *
 * Layouts: x, y (T,D) and conv_pool (num_slots,D,W-1) in dims.dtype (the state
 * holds raw inputs, exact in that dtype); weight (D,W), bias (D) fp32.  W in
 * [2, 4]; D a multiple of 8.  Read and write slots of one call are disjoint.
 * device_err (one int32 in device memory, required) receives SSD_DEVERR_*
 * bits (CU_SEQLENS, INIT_SLOT, FINAL_SLOT).  With T = 0, x and y may be NULL.
 * One launch on `stream`; allocates nothing. */
typedef struct ssd_conv_dims {
    int64_t T;          /* total tokens, >= 0 */
    int32_t R;          /* requests, >= 1 */
    int32_t D;          /* channels, a multiple of 8 */
    int32_t W;          /* kernel width, 2..4 */
    int32_t dtype;      /* enum ssd_dtype of x, y and conv_pool */
    int32_t num_slots;  /* rows of conv_pool (0 when no slots are used) */
    int32_t silu;       /* 1: SiLU activation, 0: none */
} ssd_conv_dims;

typedef struct ssd_conv_io {
    const void *x;              /* (T,D) */
    const float *weight;        /* (D,W) */
    const float *bias;          /* (D) or NULL */
    void *conv_pool;            /* (num_slots,D,W-1), or NULL when no slots are given */
    const int32_t *read_slots;  /* (R) or NULL */
    const int32_t *write_slots; /* (R) or NULL */
    void *y;                    /* (T,D) */
    int32_t *device_err;        /* one int32, OR-ed with SSD_DEVERR_* bits */
} ssd_conv_io;

int ssd_varlen_conv1d(const ssd_conv_dims *dims, const int32_t *cu_seqlens, const ssd_conv_io *io,
                      cudaStream_t stream);

/* ---- Gated delta rule (GDN) chunked prefill with state export --------------
 * "Automatic prefix caching for GDN hybrid models (mamba_cache_mode=all) with
 * MTP speculative decoding", Purpose (Kernels/layers): the gated-delta-rule
 * layers of GDN hybrid models run through a chunk kernel that exports per-chunk
 * intermediate states, checkpointed by the same block-aligned scatter as the
 * Mamba2 path.  The pages print no formula; this is the published gated delta
 * rule ("Gated Delta Networks: Improving Mamba2 with Delta Rule"), state S a
 * K x V matrix per value head h, key head h / (Hv/Hk), per token t in order:
 *     q~, k~ = q_t, k_t   (or x / sqrt(|x|^2 + 1e-6) each, when dims.l2norm)
 *     S  <- exp(g_t) S;   u = beta_t (v_t - S^T k~);   S <- S + k~ u^T
 *     o_t = scale * S^T q~
 * with S from state_pool[init_slots[i]] (zeros when < 0 or NULL).  Chunks are
 * cut at absolute multiples of chunk_size (positions counted from
 * num_computed[i]); state outputs follow the forward's rules: chunk_states row
 * first_chunk[i] + j = the state after chunk j (rows as
 * ssd_varlen_count_chunks with chunk_size), block checkpoints through
 * block_table (state after absolute token kb-1 for every multiple kb of
 * block_size in (s, s+L], entries < 0 skipped), final states to final_states[i]
 * and state_pool[final_slots[i]].  An empty request's final state is its
 * initial state.
 *
 * Supported: bf16 q, k, v, o; K = 128; V a multiple of 32 up to 256;
 * chunk_size = 64; block_size a multiple of 64 (or 0 without a block table).
 * g and beta fp32, g <= 0 expected (a decay).  With T = 0 (every request empty)
 * the token buffers may be NULL.  Write slots must not alias read
 * slots of the same call.  Host-visible violations return SSD_ERR_* before any
 * launch; device_err (one int32, required) receives SSD_DEVERR_* bits
 * (CU_SEQLENS, NUM_COMPUTED, INIT_SLOT, FINAL_SLOT, BLOCK_SLOT, BLOCK_TABLE),
 * the offending writes skipped.  One launch on `stream`; allocates nothing. */
typedef struct ssd_gdn_dims {
    int64_t T;               /* total tokens, >= 0 */
    int32_t R;               /* requests, >= 1 */
    int32_t Hk, Hv;          /* key heads, value heads (a multiple of Hk) */
    int32_t K, V;            /* key and value head dims */
    int32_t chunk_size;      /* 64 */
    int32_t block_size;      /* block-checkpoint granularity, or 0 */
    int32_t block_table_width;
    int32_t dtype;           /* enum ssd_dtype of q, k, v and o */
    int32_t num_slots;       /* rows of state_pool (0 without a pool) */
    int32_t l2norm;          /* 1: q and k l2-normalised per token inside the kernel */
    float scale;             /* output scale; 0 means K^-1/2 */
} ssd_gdn_dims;

typedef struct ssd_gdn_io {
    const void *q, *k;           /* (T,Hk,K) */
    const void *v;               /* (T,Hv,V) */
    const float *g;              /* (T,Hv) log decay per token and value head */
    const float *beta;           /* (T,Hv) write strength */
    const int32_t *num_computed; /* (R) tokens already in each request's state, or NULL */
    float *state_pool;           /* (num_slots,Hv,K,V) fp32, or NULL */
    const int32_t *init_slots;   /* (R) or NULL */
    const int32_t *final_slots;  /* (R) or NULL */
    const int32_t *block_table;  /* (R, block_table_width) or NULL */
    void *o;                     /* (T,Hv,V) */
    float *final_states;         /* (R,Hv,K,V) or NULL */
    float *chunk_states;         /* (n_chunks,Hv,K,V) or NULL */
    int32_t *device_err;         /* one int32, OR-ed with SSD_DEVERR_* bits */
} ssd_gdn_io;

int ssd_varlen_gdn_forward(const ssd_gdn_dims *dims, const int32_t *cu_seqlens, const ssd_gdn_io *io,
                           cudaStream_t stream);

/* ---- Slot aliasing check (for debug runs) ------------------------------------
 * The calls above require that no pool slot written in a call is also read in
 * it, and that no slot is written twice (the caller's responsibility: checking
 * it on every call would cost a pass over the slot tables).  This entry point
 * checks it on the device, for debug runs: with R = dims->R requests,
 *   read slots  = init_slots[i] >= 0
 *   write slots = final_slots[i] >= 0 and block_table[i][j] >= 0
 *                 (j < dims->block_table_width)
 * it ORs SSD_DEVERR_ALIAS into *device_err when a write slot equals a read slot
 * or another write slot (the decode step's anchors: pass read_slots as
 * init_slots and its per-token write_slots as final_slots with R = T).  Any of
 * the three tables may be NULL.  O((R + R W)^2) comparisons on the device: meant
 * for tests and debug builds, not for every step.  One launch on `stream`;
 * allocates nothing.  Returns SSD_ERR_NULL without device_err, SSD_ERR_DIMS for
 * R < 1 or a negative width. */
int ssd_varlen_check_slots(const ssd_dims *dims, const int32_t *init_slots, const int32_t *final_slots,
                           const int32_t *block_table, int32_t *device_err, cudaStream_t stream);

/* ---- Block-aligned prefill bites (host only) --------------------------------
 * "Automatic prefix caching for GDN hybrid models (mamba_cache_mode=all) with
 * MTP speculative decoding", Purpose (engine core: kernel-chunk-aligned prefill
 * clipping and block-aligned split in the scheduler) and the review note on
 * that page about re-aligning a misaligned start in the final bite.
 * A scheduler proposes to prefill positions [start, end) of a prompt that ends
 * at `total`; the bite is clipped so that the next bite starts on the align
 * grid (align = the block size, a multiple of chunk_size).  With
 * last_aligned = total rounded down to a multiple of align:
 *   - a start off the grid ends the bite at the next boundary, when that
 *     boundary is at most last_aligned (also in the final bite);
 *   - otherwise an end before last_aligned is rounded down to a boundary, which
 *     is start itself when the budget is below one block: the request then
 *     waits for a step with a larger budget;
 *   - an aligned start reaching last_aligned may end anywhere (the tail).
 * Returns the clipped end (start <= result <= end), or SSD_ERR_DIMS (< 0) when
 * align < 1, start < 0, end <= start or end > total.  Pure host arithmetic. */
int64_t ssd_varlen_align_bite(int64_t start, int64_t end, int64_t total, int32_t align);

#ifdef __cplusplus
}
#endif

#endif /* SSD_VARLEN_H */
