/*
 * bi_gemm.h -- C ABI of the batch-invariant bf16 linear layer (GB300, sm_103a).
 *
 * What the library computes
 *   GEMM      Y[M,N] = X[M,K] . W[N,K]^T, bf16 storage, fp32 accumulation,
 *             round-to-nearest-even to bf16 at the end.
 *   RMSNorm   y_h = bf16_rne((x_h * r) * g_h),  r = 1 / sqrt(mean_h(x_h^2) + eps),
 *             per row, with fp32 arithmetic.
 *   Fused     RMSNorm followed by the GEMM, bit for bit equal to the two calls
 *             made one after the other, with the normalisation applied to X
 *             in shared memory: the normalised rows never reach device memory.
 *   Glue      the element-wise steps of a Llama-style decode layer (residual
 *             add, SiLU(gate) * up, and the attention stand-in for a context of
 *             one token).
 *
 * Batch invariance.  Detent (Batch-Invariant LLM Serving and RL Rollouts at
 * Near-Stock Speed), Sec. 3, Eq. 2, asks that a request's output bits not
 * depend on the batch it runs in, and gives the sufficient condition (Sec. 1,
 * Eq. 1) that each kernel is batch-invariant and that kernel selection never
 * reads the batch.  CoRun (Padding is Simple and Efficient for Deterministic
 * LLM Inference), Sec. III-B, Def. 1, states the kernel contract:
 * x_i = x'_j implies F_n(X)_i = F_m(X')_j for all batch sizes n, m and rows
 * i, j.  This library meets it by construction: every output row's floating
 * point reduction tree -- the K-tile, the number of K splits and their
 * boundaries, the order in which the split partials are added, the tensor-core
 * instruction shape -- is a function of (N, K, pins) only.  M, the row's
 * position and the other rows' values choose only which SM computes what.
 *
 * Pins.  Detent, Sec. 3, calls a value of kernel selection that is replaced by
 * a constant a pin, and the set of pins fixed before serving a commitment
 * tuple; an illegal assignment stops the engine before any kernel runs
 * (Sec. 5).  bi_pins is the GEMM family's slice of such a tuple: callers fix
 * one bi_pins per (N, K) for a deployment and pass it on every call.
 * bi_pins_default() gives the library's table entry, which never reads M.
 *
 * Conventions for every entry point
 *   - Pointers are caller-owned DEVICE memory of the current CUDA device, bf16
 *     tensors row-major and contiguous, 16-byte aligned.  The library keeps no
 *     reference to them after the call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and return launch-time errors only.  A device-side
 *     stall (a bounded wait that ran out) is reported by
 *     bi_last_device_status().
 *   - Arguments are checked before anything is launched; a call that returns
 *     an error launched nothing and wrote nothing.
 *   - M == 0 is a successful no-op.
 *   - The library allocates no device memory on any call.  The fused call
 *     takes a caller-provided workspace (4 bytes per row).
 *   - Device addresses of the library's own static device variables (the
 *     stall word, the no-alloc scratch) are looked up once per device and
 *     cached; they do not survive cudaDeviceReset, after which the library
 *     must not be called again in the same process.
 *   - Entry points are reentrant; calls on different streams may overlap.
 */
#ifndef BI_GEMM_H
#define BI_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* bi_stream_t;

#define BI_PINS_ABI_VERSION 1

/* bf16 elements per K tile.  The only supported value. */
#define BI_BK 64
/* Output features (rows of W) per tensor-core tile: the MMA's M extent. */
#define BI_TILE_N 128
/* Largest number of K splits. */
#define BI_MAX_SPLIT_K 16

/* Schedule flags: speed only.  They choose how the S split chains of a tile
 * are placed on SMs and never change any output bit: the partials are always
 * added in ascending split order, ((P0 + P1) + P2) + ...
 *   AUTO     the library chooses from M (allowed: it changes no bit).
 *   LOCAL    one persistent CTA (or pair) per tile computes its S chains one
 *            after the other into two TMEM accumulators and folds them in
 *            registers.
 *   CLUSTER  a cluster of S CTAs (or pairs) computes one chain each and folds
 *            the S partials through distributed shared memory (S <= 8).
 *   CHAIN    a cluster of ceil(S/2) CTAs (or pairs) per tile; each computes
 *            two consecutive chains (one for the first when S is odd).  Each
 *            adds its chains, in order, to the running sum the previous one
 *            left in shared memory (S >= 3).
 *   GLOBAL   (bi_gemm_bf16_ws with a fold workspace; one token tile,
 *            single-CTA MMAs, 2 <= S <= 8) persistent CTAs take the S * tiles
 *            chains one by one, with no cluster co-residency limit; each
 *            chain's partial goes to the workspace, and the chain that
 *            finishes its tile's set last folds the S partials there in
 *            ascending order.  Elsewhere the flag falls back to AUTO. */
#define BI_FLAG_SCHEDULE_AUTO 0x0u
#define BI_FLAG_SCHEDULE_LOCAL 0x1u
#define BI_FLAG_SCHEDULE_CLUSTER 0x2u
#define BI_FLAG_SCHEDULE_CHAIN 0x3u
#define BI_FLAG_SCHEDULE_GLOBAL 0x4u
#define BI_FLAG_SCHEDULE_MASK 0x7u
/* Splits the GLOBAL schedule folds at most. */
#define BI_GLOBAL_MAX_SPLIT_K 8
/* Diagnostic only: the load producer withholds its first load so that the
 * tensor-core warp's bounded wait runs out.  The kernel then abandons the call
 * (Y is left unspecified), frees its tensor memory and returns, and
 * bi_last_device_status() reports BI_ERR_DEVICE_TIMEOUT.  Exists to test the
 * stall detection; never set it otherwise. */
#define BI_FLAG_DEBUG_STALL_PRODUCER 0x100u
/* Speed only.  Every kernel of this library is launched so that it may start
 * while the previous kernel in the stream is still finishing; it waits for that
 * kernel before reading any input or writing any output.  With this flag the
 * GEMM also starts streaming W before that wait, so a decode step's weight
 * stream overlaps the small kernels before it.  The caller must then guarantee
 * that W is not written by any kernel still running in the stream when the
 * call is made (weights are normally written once, long before). */
#define BI_FLAG_PREFETCH_W 0x200u
/* Speed only.  Copy W and X two K tiles at a time into ring stages of two K
 * tiles (through 3-D views of the matrices), so that the tensor-core warp
 * waits and commits once per eight MMAs instead of four.  Honoured when
 * K % 64 == 0, tok_tile == 256 and the X copies cover the whole token tile;
 * otherwise one K tile per copy.  The MMAs consume K tiles one by one in the
 * same order either way, so the flag never changes a bit of Y. */
#define BI_FLAG_KTILE_PAIRS 0x400u
/* Speed only, read by the fused call (bi_rmsnorm_gemm_bf16 and its no-alloc
 * form) alone.  The fused call applies the RMSNorm to X in one of two ways,
 * with the same bits: staged, the standalone RMSNorm kernel writing the
 * normalised rows to the workspace for the GEMM to read (the default), or in
 * shared memory, as each X tile arrives for the tensor cores, so that the
 * normalised rows never reach device memory.  In shared memory the
 * normalisation is repeated for every W tile that meets an X tile, and each
 * CTA's first stage waits for the rows' scales; measured on GB300 it is the
 * slower form at every batch size of the Llama-3.1-8B projections (by about
 * 2% at one token, 3x at thousands), so it is used only when forced
 * (BI_FLAG_NORM_SMEM) or when the no-alloc call has no room to stage.  Both
 * flags set: illegal. */
#define BI_FLAG_NORM_SMEM 0x800u
#define BI_FLAG_NORM_STAGED 0x1000u
#define BI_FLAG_KNOWN_MASK                                                                              \
  (BI_FLAG_SCHEDULE_MASK | BI_FLAG_DEBUG_STALL_PRODUCER | BI_FLAG_PREFETCH_W | BI_FLAG_KTILE_PAIRS | \
   BI_FLAG_NORM_SMEM | BI_FLAG_NORM_STAGED)

typedef struct bi_pins {
  int32_t abi_version; /* BI_PINS_ABI_VERSION */
  int32_t bk;          /* K-tile width in bf16 elements: BI_BK */
  int32_t split_k;     /* S, the number of K splits, 1..BI_MAX_SPLIT_K and at most
                          the number of K tiles.  Split s covers K tiles
                          [floor(s*KT/S), floor((s+1)*KT/S)), KT = ceil(K/bk); the
                          partials are added in ascending s. */
  int32_t tok_tile;    /* T, tokens per tile = the MMA's N extent: 64, 128 or 256 */
  int32_t mma_ctas;    /* 1: tcgen05.mma.cta_group::1, 128 W rows per MMA;
                          2: tcgen05.mma.cta_group::2 across a CTA pair, 256 W rows
                          per MMA (each CTA holds 128 W rows and T/2 tokens);
                          0: chosen per launch for speed.  Both groupings give
                          every output element the same bits (each is one chain
                          of k16 steps in the same order), which the GPU tests
                          check; pin 1 or 2 to fix the grouping regardless. */
  int32_t stages;      /* depth of the W shared-memory ring, in copies (a copy
                          holds bi_gemm_plan.kps K tiles); 0 = chosen by the
                          library from the launch.  Speed only. */
  uint32_t flags;      /* BI_FLAG_* */
} bi_pins;

typedef enum bi_status {
  BI_OK = 0,
  BI_ERR_INVALID_ARG = 1,       /* NULL pointer, negative size, bad eps, ... */
  BI_ERR_ALIGNMENT = 2,         /* a pointer not 16-byte aligned */
  BI_ERR_UNSUPPORTED_SHAPE = 3, /* e.g. K not a multiple of 8, a dimension too large */
  BI_ERR_ILLEGAL_PINS = 4,      /* bi_pins_validate() refused the pins */
  BI_ERR_CUDA = 5,              /* a CUDA runtime call failed (launch, no device, ...) */
  BI_ERR_DEVICE_TIMEOUT = 6,    /* a kernel's bounded wait ran out (see bi_last_device_status) */
  BI_ERR_WORKSPACE = 7,         /* workspace missing or smaller than required */
  BI_ERR_DEBUG_BOUNDS = 8       /* (debug-bounds build only) a kernel's index check failed; the
                                   access was skipped (see bi_debug_bounds_detail) */
} bi_status;

/* Version of this ABI (BI_PINS_ABI_VERSION). */
int32_t bi_abi_version(void);

/* Human-readable name of a status.  Never NULL; static storage. */
const char* bi_status_string(bi_status status);

/* 1 in the debug-bounds build of the library (libbi_gemm_debug.so, compiled
 * with -DBI_DEBUG_BOUNDS), 0 in the ordinary one.  In the debug-bounds build
 * the GEMM and decode-attention kernels check, before each access, their tile
 * coordinates (W and X rows, K tiles) and their ring-stage, tensor-memory
 * column, fold-workspace and split-record indices against the bounds of what
 * they address.  A failed check skips the access (it never traps), records
 * BI_ERR_DEBUG_BOUNDS for bi_last_device_status(), and keeps the first
 * failure's check number and value for bi_debug_bounds_detail(); the kernel
 * then gives up through its bounded waits.  Same ABI and same bits otherwise:
 * a speed-only variant for tests.  Host only. */
int32_t bi_debug_bounds_enabled(void);

/* The first failed check since the last call, as (check << 48) | value, and
 * clears it (0 when none failed).  The check numbers are listed in the
 * library's bounds.cuh.  Synchronises `stream`.  Errors: BI_ERR_INVALID_ARG
 * (detail NULL), BI_ERR_CUDA. */
bi_status bi_debug_bounds_detail(uint64_t* detail, bi_stream_t stream);

/* The library's pins for a GEMM with N output features and reduction length
 * K.  There is no M argument: the table is keyed on (N, K) alone (Detent,
 * Sec. 8.2: the batch reaches neither GEMM selection point).  Fills *out.
 * Errors: BI_ERR_INVALID_ARG (out NULL, N or K < 1),
 * BI_ERR_UNSUPPORTED_SHAPE (K % 8 != 0).  Host only; touches no GPU. */
bi_status bi_pins_default(int64_t N, int64_t K, bi_pins* out);

/* Checks pins for (N, K): version, bk == BI_BK, 1 <= split_k <= min(16, KT),
 * tok_tile in {64,128,256}, mma_ctas in {1,2}, stages 0 or in the legal range,
 * flags known, CLUSTER only with split_k <= 8.  Returns BI_OK or
 * BI_ERR_ILLEGAL_PINS (BI_ERR_INVALID_ARG for a NULL pointer).  Host only. */
bi_status bi_pins_validate(int64_t N, int64_t K, const bi_pins* pins);

/* A description of the launch the GEMM would make, for inspection and tests.
 * Reduction tree (bk, split_k, mma_k, k_tiles, split_begin): a function of
 * (N, K, pins) only.  MMA layout (tok_tile, mma_ctas, mma_m, mma_n): how many
 * output elements one MMA computes side by side, and on how many SMs; fixed
 * by the pins when they fix mma_ctas, chosen per launch when mma_ctas = 0.  It
 * never changes a bit of Y.  Everything else is the schedule and may depend
 * on M. */
typedef struct bi_gemm_plan {
  int32_t bk, split_k;                     /* tree */
  int32_t tok_tile, mma_ctas, mma_m, mma_n; /* MMA layout */
  int32_t mma_k;                           /* tree: 16 K elements per MMA step */
  int64_t k_tiles;                         /* tree */
  int64_t split_begin[BI_MAX_SPLIT_K + 1]; /* tree: K-tile boundaries, split s = [begin[s], begin[s+1]) */
  /* schedule: may depend on M */
  int32_t schedule;                        /* BI_FLAG_SCHEDULE_LOCAL, _CLUSTER, _CHAIN or _GLOBAL */
  int32_t units;                           /* cluster schedules: CTAs (or pairs) per tile */
  int32_t w_stages, x_stages;              /* depths of the W and X shared-memory rings */
  int32_t x_box_rows;                      /* token rows per X copy (< tok_tile for small M) */
  int32_t kps;                             /* K tiles per copy and ring stage (1, or 2 with
                                              BI_FLAG_KTILE_PAIRS and paired MMAs).  The MMAs
                                              consume the K tiles one by one, in order, either
                                              way. */
  int64_t n_tiles, m_tiles;
  int32_t group_n;                         /* LOCAL tile order: W tiles per group (0 for CLUSTER) */
  int32_t grid_x, grid_y, grid_z, cluster_x, block_threads;
  int64_t smem_bytes;
} bi_gemm_plan;

/* Fills *plan for a GEMM of shape (M, N, K) with the given pins (NULL = the
 * default pins).  `sm_count` sizes the persistent grid (0 = 152, the SM count
 * of a GB300); it never changes the tree fields.  Host only.
 * Errors: as bi_gemm_bf16's argument checks. */
bi_status bi_gemm_plan_describe(int64_t M, int64_t N, int64_t K, const bi_pins* pins,
                                int32_t sm_count, bi_gemm_plan* plan);

/* Y[M,N] = bf16_rne(X[M,K] . W[N,K]^T), fp32 accumulation on the tensor cores.
 *   X  [M,K] bf16 activations (tokens), W [N,K] bf16 weights, Y [M,N] bf16 out.
 *   pins NULL = bi_pins_default(N, K).
 * Requirements: K % 8 == 0 (16-byte row pitch for the tensor-memory copies),
 * X, W, Y 16-byte aligned, M, N, K < 2^31.
 * Defines: LLM-42 (Enabling Determinism in LLM Inference with Verified
 * Speculation), Sec. 2.2, Fig. 3: a GEMM whose split-K use follows the shape
 * changes a token's reduction tree; here S and the split boundaries are pins.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_ALIGNMENT, BI_ERR_UNSUPPORTED_SHAPE,
 * BI_ERR_ILLEGAL_PINS, BI_ERR_CUDA. */
bi_status bi_gemm_bf16(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                       const bi_pins* pins, bi_stream_t stream);

/* Bytes of fold workspace bi_gemm_bf16_ws can use for this call: the GLOBAL
 * schedule's per-tile arrival counters (the first 256-byte-rounded
 * ceil(N/128) * 4 bytes) and chain partials (ceil(N/128) * S * T * 128 * 4
 * bytes, T the launch's token tile).  0 when the GLOBAL schedule does not
 * apply (more than one token tile, paired MMAs, S outside 2..8), or on
 * invalid arguments.  Host only. */
size_t bi_gemm_bf16_workspace_bytes(int64_t M, int64_t N, int64_t K, const bi_pins* pins);

/* bi_gemm_bf16 with a fold workspace: the same bits for the same pins (the
 * tree never depends on the schedule), and one more schedule the planner may
 * choose for a single token tile (decode): GLOBAL (see the schedule flags).
 * It puts a tile's S split chains on any SMs with no cluster co-residency
 * limit, so a decode step streams W through every SM.
 * Workspace: caller-owned device memory of at least
 * bi_gemm_bf16_workspace_bytes(M, N, K, pins) bytes (smaller or NULL: the
 * call runs as bi_gemm_bf16), 256-byte aligned.  Its counter part must be
 * zero before the first call (cudaMemset); every call that completes leaves
 * it zero again, so a workspace is zeroed once.  A call abandoned by a
 * bounded wait (BI_ERR_DEVICE_TIMEOUT) may leave counts behind: zero it
 * again.  Calls that may overlap on the GPU need workspaces of their own.
 * Defines: LLM-42, Sec. 2.2, Fig. 3 and CoRun, Sec. III-A, Fig. 3(b): the
 * split count and the order in which split partials are added are fixed by
 * (N, K, pins); here they are added in ascending split order wherever they
 * are folded.
 * Errors: as bi_gemm_bf16, plus BI_ERR_ALIGNMENT for the workspace. */
bi_status bi_gemm_bf16_ws(const void* X, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                          const bi_pins* pins, void* workspace, size_t workspace_bytes, bi_stream_t stream);

/* As bi_gemm_plan_describe, for bi_gemm_bf16_ws with a workspace of
 * `workspace_bytes` bytes. */
bi_status bi_gemm_plan_describe_ws(int64_t M, int64_t N, int64_t K, const bi_pins* pins, int32_t sm_count,
                                   size_t workspace_bytes, bi_gemm_plan* plan);

/* Bytes of device workspace bi_gemm_bf16_host needs for M rows (0 for M = 0):
 * a ring of two chunk slots, or one when one chunk holds every row. */
size_t bi_gemm_bf16_host_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Y_host[M,N] = bf16(X_host[M,K] . W[N,K]^T) with X and Y in host memory and W
 * on the device: the same bits as bi_gemm_bf16 on device copies of X and Y.
 * The rows travel in chunks of about 16 MB of X through a ring of buffers in
 * `workspace`: a chunk is copied in on a library stream, multiplied on
 * `stream` and copied out on a second library stream, so copies and GEMMs of
 * consecutive chunks overlap.  Chunking is free because the tree of a row
 * never depends on M (Detent, Sec. 3: a batch-invariant operator gives each
 * row the same bits whatever batch it is computed in).
 * Ring depth: as many slots of bi_gemm_bf16_host_slot_bytes bytes as
 * `workspace_bytes` holds, at most 8 and at most the number of chunks; the
 * size the workspace query returns gives two.  With three or more slots the
 * last rows go in halving chunks (multiples of 128 rows, the last 256 or
 * fewer whole), so that little is left to multiply and copy out after the
 * last copy-in.
 * Ownership: X_host and Y_host are caller-owned host memory (page-locked for
 * the copies to overlap; pageable memory works, with synchronous copies);
 * W and `workspace` are caller-owned device memory, `workspace` at least
 * bi_gemm_bf16_host_workspace_bytes(M, N, K) bytes and 256-byte aligned, not
 * used by work that is not ordered before this call on `stream`.  The library
 * keeps two streams and a few events per device, created on first use.
 * Asynchrony: the call enqueues its work after everything already on
 * `stream`, and `stream` waits for the last rows to reach Y_host; synchronize
 * `stream` before reading Y_host.
 * Requirements: as bi_gemm_bf16 (W 16-byte aligned; X_host and Y_host need no
 * alignment).
 * Errors: as bi_gemm_bf16, plus BI_ERR_WORKSPACE.  Every argument is checked
 * before any work is enqueued. */
bi_status bi_gemm_bf16_host(const void* X_host, const void* W, void* Y_host, int64_t M, int64_t N, int64_t K,
                            const bi_pins* pins, void* workspace, size_t workspace_bytes, bi_stream_t stream);

/* One job of bi_gemm_bf16_host_batch: Y_host[M,N] = X_host[M,K] . W[N,K]^T. */
typedef struct bi_host_gemm_job {
  const void* X_host; /* [M, K] bf16, row-major, host memory */
  const void* W;      /* [N, K] bf16, row-major, device memory, 16-byte aligned */
  void* Y_host;       /* [M, N] bf16, row-major, host memory */
  int64_t M;          /* rows; 0 skips the job (its pointers may then be NULL) */
} bi_host_gemm_job;

/* Bytes of device workspace bi_gemm_bf16_host_batch needs for `jobs` and
 * `chunk_rows` (0 when no job has rows, or for an invalid argument): two
 * chunk slots, or one when one chunk holds every row of every job. */
size_t bi_gemm_bf16_host_batch_workspace_bytes(const bi_host_gemm_job* jobs, int32_t n_jobs, int64_t N, int64_t K,
                                               int64_t chunk_rows);

/* Bytes of one ring slot (a chunk's X and Y) for `jobs` and `chunk_rows`; a
 * workspace of d slots gives a ring of depth d (at most 8).  With one job of
 * M rows and chunk_rows 0 this is the slot of bi_gemm_bf16_host. */
size_t bi_gemm_bf16_host_slot_bytes(const bi_host_gemm_job* jobs, int32_t n_jobs, int64_t N, int64_t K,
                                    int64_t chunk_rows);

/* The GEMMs of a list of jobs of one shape (N, K) and one set of pins, with X
 * and Y in host memory: each job gives the bits bi_gemm_bf16 gives on device
 * copies of its X and Y.  The jobs' rows run as one sequence of chunks through
 * one ring, in job order, so the copies of one job overlap the GEMMs of its
 * neighbours as they overlap those of its own chunks (Detent, Sec. 3: the
 * bits of a row do not depend on the launch it is computed in).  The jobs may
 * share W or not.
 * chunk_rows: rows per chunk (capped at the largest job's rows); 0 takes the
 * rule of bi_gemm_bf16_host for the largest job (about 16 MB of X, a multiple
 * of 128 rows).  Larger chunks run the GEMMs faster and stretch the last
 * chunk's GEMM and copy-out; the chunk size changes no bit.
 * Ownership, asynchrony and the ring depth: as bi_gemm_bf16_host, with
 * `workspace` at least bi_gemm_bf16_host_batch_workspace_bytes bytes.  The
 * job array itself is read during the call only.
 * Errors: BI_ERR_INVALID_ARG for n_jobs < 0, a NULL `jobs` with n_jobs > 0, a
 * negative M or chunk_rows, or a NULL pointer of a job with rows;
 * BI_ERR_UNSUPPORTED_SHAPE for chunk_rows above 2^31 - 1; otherwise as
 * bi_gemm_bf16_host.  Every argument is checked before any work is enqueued. */
bi_status bi_gemm_bf16_host_batch(const bi_host_gemm_job* jobs, int32_t n_jobs, int64_t N, int64_t K,
                                  const bi_pins* pins, int64_t chunk_rows, void* workspace, size_t workspace_bytes,
                                  bi_stream_t stream);

/* One chunk of the schedule bi_gemm_bf16_host_batch follows. */
typedef struct bi_host_chunk {
  int32_t job;  /* index of the job in the list */
  int32_t slot; /* ring slot holding the chunk's X and Y */
  int64_t row0; /* first row of the job in the chunk */
  int64_t rows; /* rows in the chunk */
} bi_host_chunk;

/* The chunk schedule of bi_gemm_bf16_host_batch for these arguments (only
 * each job's M is read): the chunks in the order they are copied in,
 * multiplied and copied out, each job's rows covered once and in order.
 * Writes the first min(*n_chunks, max_chunks) chunks to `chunks` and the
 * count to *n_chunks (0 when no job has rows).  A host-only call.
 * Errors: BI_ERR_INVALID_ARG for a NULL n_chunks, max_chunks < 0 or a NULL
 * `chunks` with max_chunks > 0; BI_ERR_WORKSPACE for workspace_bytes below
 * bi_gemm_bf16_host_batch_workspace_bytes; otherwise as
 * bi_gemm_bf16_host_batch for the rows, the shape and chunk_rows. */
bi_status bi_gemm_bf16_host_schedule(const bi_host_gemm_job* jobs, int32_t n_jobs, int64_t N, int64_t K,
                                     int64_t chunk_rows, size_t workspace_bytes, bi_host_chunk* chunks,
                                     int64_t max_chunks, int64_t* n_chunks);

/* Y[M,H] = RMSNorm(X[M,H]) with gain g[H], one warp per row: each lane sums
 * the squares of its 16-byte vectors in ascending order, the 32 lane sums are
 * combined by a fixed xor-butterfly, r = 1/sqrt(sum/H + eps) (IEEE division
 * and square root), y = bf16_rne((x * r) * g).  The tree depends on H only.
 * Defines: LLM-42, Sec. 2.1 (normalisation reduces over the hidden dimension
 * of each token); CoRun, Fig. 2(a) (RMSNorm among the batch-invariant
 * operators).
 * Requirements: H % 8 == 0, 8 <= H <= 65536, eps > 0 and finite, pointers
 * 16-byte aligned.  X and Y may be the same buffer.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_ALIGNMENT, BI_ERR_UNSUPPORTED_SHAPE,
 * BI_ERR_CUDA. */
bi_status bi_rmsnorm_bf16(const void* X, const void* g, void* Y, int64_t M, int64_t H, float eps,
                          bi_stream_t stream);

/* Bytes of workspace bi_rmsnorm_gemm_bf16 needs for M rows of width K: one
 * fp32 value per row, then room for the normalised rows [M,K] bf16 (used by
 * the staged form only), each part rounded up to 256 bytes.  0 for M = 0. */
size_t bi_rmsnorm_gemm_workspace_bytes(int64_t M, int64_t K);

/* Y = bi_gemm_bf16(bi_rmsnorm_bf16(X; g, eps), W), bit for bit, with
 * X [M,K] the raw activations, g [K] the gain, W [N,K], Y [M,N]; H of the
 * RMSNorm is K.
 * Defines: LLM-42 (Enabling Determinism in LLM Inference with Verified
 * Speculation), Sec. 2.1: the normalisation reduces over the hidden dimension
 * of each token, so it is row-local and its tree depends on K alone; the
 * fused layer is read as the composition of the two batch-invariant
 * operators, through the bf16 normalised rows.
 * How: by default the standalone RMSNorm kernel writes the normalised rows
 * to the workspace and the GEMM reads them (the two calls in sequence, on
 * the caller's stream).  With BI_FLAG_NORM_SMEM, r[m] = 1 / sqrt(mean(x^2) +
 * eps) of each row is computed first with the RMSNorm's lane partition and
 * butterfly (the same bits; by the GEMM itself for at most 4 rows, else by a
 * row-scale kernel), and the GEMM applies bf16_rne((x * r[m]) * g[k]) to each
 * X tile in shared memory between its arrival and the tensor-core reads, so
 * the normalised rows never reach device memory.  Both forms give the same
 * bits.
 * Workspace: caller-owned device memory, 256-byte aligned, of at least
 * bi_rmsnorm_gemm_workspace_bytes(M, K) bytes: the RMSNorm's scratch (r and
 * the staged rows), taken from the workspace's end; its contents there on
 * return are unspecified.  Bytes in front of that part serve as the GEMM's
 * fold workspace (as for bi_gemm_bf16_ws) when there are at least
 * bi_gemm_bf16_workspace_bytes(M, N, K, pins) of them: then the workspace's
 * first bytes hold the fold counters, which must be zero before the first
 * call and which every completed call leaves zero.  The library allocates
 * nothing, so the caller provides it; bi_rmsnorm_gemm_bf16_noalloc takes none.
 * Errors: as the two calls, plus BI_ERR_WORKSPACE.  Everything is checked and
 * the GEMM planned before the first kernel is launched. */
bi_status bi_rmsnorm_gemm_bf16(const void* X, const void* g, const void* W, void* Y, int64_t M,
                               int64_t N, int64_t K, float eps, const bi_pins* pins,
                               void* workspace, size_t workspace_bytes, bi_stream_t stream);

/* Capacity in bytes of the static scratch array used by
 * bi_rmsnorm_gemm_bf16_noalloc: r takes 4 bytes per row (rounded up to 256),
 * so M may not exceed 4194240; the staged form also needs M * K * 2 bytes. */
#define BI_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)

/* BI_NOALLOC_SCRATCH_BYTES as compiled into the library (for bindings that
 * do not read this header). */
size_t bi_noalloc_scratch_bytes(void);

/* The fused layer for callers that cannot allocate device memory -- for
 * example a plugin inside a host runtime that has reserved the device's memory
 * and offers no allocator, or a latency-critical path where cudaMalloc /
 * cudaFree would synchronise the device.  Same arguments, result and bits as
 * bi_rmsnorm_gemm_bf16, but no workspace: the per-row RMSNorm scales (and
 * the staged normalised rows, when that form is used) are kept in a static
 * device array of BI_NOALLOC_SCRATCH_BYTES that the library holds on every
 * GPU that loads it, until the process exits.  Where the staged rows would
 * not fit, the rows are normalised in shared memory instead (same bits).  The
 * call allocates nothing.
 *   - The first call on a device looks the array's address up (with that
 *     device current) and caches it; make that first call before any stream
 *     capture.  The cache does not survive cudaDeviceReset.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents; calls whose work overlaps on the GPU (e.g. on two streams)
 *     race on it and must be serialised by the caller.
 * Errors: as bi_rmsnorm_gemm_bf16; BI_ERR_WORKSPACE when M * 4 (rounded up
 * to 256) exceeds BI_NOALLOC_SCRATCH_BYTES (nothing is launched).
 * The paper has no counterpart to this entry point. */
bi_status bi_rmsnorm_gemm_bf16_noalloc(const void* X, const void* g, const void* W, void* Y,
                                       int64_t M, int64_t N, int64_t K, float eps,
                                       const bi_pins* pins, bi_stream_t stream);

/* out[i] = bf16_rne(float(a[i]) + float(b[i])) for i < count (the residual
 * connection of a decode layer).  count % 8 == 0, pointers 16-byte aligned;
 * out may alias a or b. */
bi_status bi_residual_add_bf16(const void* a, const void* b, void* out, int64_t count,
                               bi_stream_t stream);

/* SwiGLU activation: gu [M, 2I] holds gate (columns 0..I-1) and up (columns
 * I..2I-1); out[m,i] = bf16_rne(silu(gate) * up) with silu(v) = v / (1 +
 * exp(-v)) in fp32.  I % 8 == 0, pointers 16-byte aligned. */
bi_status bi_silu_mul_bf16(const void* gu, void* out, int64_t M, int64_t I, bi_stream_t stream);

/* Attention at a context of one token: qkv [M, (nq + 2 nkv) D] is
 * [q | k | v]; with a single key the softmax weight is exactly 1, so query
 * head j outputs the v vector of group j / (nq / nkv).  out [M, nq D].
 * nq % nkv == 0, D % 8 == 0, pointers 16-byte aligned. */
bi_status bi_attention_ctx1_bf16(const void* qkv, void* out, int64_t M, int64_t nq, int64_t nkv,
                                 int64_t D, bi_stream_t stream);

/* ---- FP8 (E4M3) with per-token and per-channel scales ---------------------
 * Detent (Batch-Invariant LLM Serving and RL Rollouts at Near-Stock Speed),
 * Limits: dynamic per-tensor FP8 activation scales span the batch; per-token
 * (or static) scales keep each row's bits its own.  The pages give no format:
 * E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest finite
 * value 448, no infinities) with a per-row scale amax / 448. */

/* Per-row quantisation: for each row of X [M,K] bf16, amax = max |x|,
 * scale[m] = amax / 448 and inv = 448 / amax (IEEE divisions, once per row;
 * both 1 for a zero row; inv clamped to the largest finite float when 448 / amax
 * overflows), Q[m,k] = E4M3(x * inv), the fp32 product rounded to
 * nearest even, saturated at +-448.  A row with
 * a NaN or an infinity gets scale NaN and NaN codes (0x7F).  Used for the
 * activations (per token) and, offline, for the weights (per output channel).
 * Q: uint8 [M,K]; scale: fp32 [M].
 * Requirements: K % 16 == 0, X and Q 16-byte aligned, scale 4-byte aligned.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_ALIGNMENT, BI_ERR_UNSUPPORTED_SHAPE,
 * BI_ERR_CUDA. */
bi_status bi_quantize_rows_e4m3(const void* X, void* Q, float* scale, int64_t M, int64_t K,
                                bi_stream_t stream);

/* RMSNorm and per-row quantisation in one call: Q and scale are those of
 * bi_quantize_rows_e4m3 applied to Y = bi_rmsnorm_bf16(X; g, eps), bit for
 * bit (the same RMSNorm tree and rounding, the same amax, scale and codes),
 * but X is read once and Y never reaches memory.  The FP8 form of the RMSNorm
 * prologue.  Defines: LLM-42, Sec. 2.1 (the per-token normalisation) and
 * Detent, Limits (per-token scales).
 * X [M,H] bf16, g [H] bf16; Q: uint8 [M,H]; scale: fp32 [M].
 * Requirements: H % 16 == 0, 16 <= H <= 16384, eps > 0 and finite, X, g and Q
 * 16-byte aligned, scale 4-byte aligned.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_ALIGNMENT, BI_ERR_UNSUPPORTED_SHAPE,
 * BI_ERR_CUDA. */
bi_status bi_rmsnorm_quantize_e4m3(const void* X, const void* g, void* Q, float* scale, int64_t M, int64_t H,
                                   float eps, bi_stream_t stream);

/* Pins of the FP8 GEMM: as bi_pins_default / bi_pins_validate with bk = 128
 * (a K tile is 128 E4M3 values, the same 128 bytes) and tok_tile = 256. */
bi_status bi_pins_default_fp8(int64_t N, int64_t K, bi_pins* out);
bi_status bi_pins_validate_fp8(int64_t N, int64_t K, const bi_pins* pins);
bi_status bi_gemm_plan_describe_fp8(int64_t M, int64_t N, int64_t K, const bi_pins* pins,
                                    int32_t sm_count, bi_gemm_plan* plan);

/* Y[M,N] = bf16_rne((acc[m,n] * sx[m]) * sw[n]),  acc = Xq . Wq^T with fp32
 * accumulation on the tensor cores (tcgen05.mma kind::f8f6f4, 32 K values per
 * step).  Xq [M,K] and Wq [N,K] are E4M3 codes (bi_quantize_rows_e4m3), sx [M]
 * and sw [N] their scales.  The reduction tree is the bf16 GEMM's -- K tiles,
 * split count and boundaries, fold order, all fixed by (N, K, pins) -- and the
 * scales touch only the finished sum of their own row and column.
 * Requirements: K % 16 == 0, Xq, Wq, Y 16-byte aligned, sx and sw 4-byte
 * aligned, M, N, K < 2^31.  pins NULL = bi_pins_default_fp8(N, K).
 * Errors: as bi_gemm_bf16. */
bi_status bi_gemm_fp8(const void* Xq, const float* sx, const void* Wq, const float* sw, void* Y,
                      int64_t M, int64_t N, int64_t K, const bi_pins* pins, bi_stream_t stream);

/* ---- Decode attention over a paged key/value cache -----------------------
 * Detent (Batch-Invariant LLM Serving and RL Rollouts at Near-Stock Speed),
 * Sec. 7 (Kernels): attention keeps split-KV, but a request's split
 * boundaries follow a fixed split size, so they never depend on the batch.
 * LLM-42, Sec. 4.4, and CoRun, Sec. IV-B, name the alternative, no split at
 * all.  The split size is the pin: fix one per deployment and pass it on
 * every call, as with bi_pins. */
#define BI_ATTN_HEAD_DIM 128
#define BI_ATTN_MAX_SPLIT 4096
#define BI_ATTN_DEFAULT_SPLIT 256

/* Workspace of bi_decode_attention_bf16, in *bytes: 256 + the item list
 * (B * n_split * 4, rounded up to 256) + B * Hkv * n_split * (128 + 2) * GP * 4,
 * n_split = max(1, ceil(max_seq_len / split_size)), GP = 8 for up to 8 query
 * heads per key/value head, else 16.  split_size 0 = BI_ATTN_DEFAULT_SPLIT.
 * Every call rewrites the whole workspace it uses: no initial contents are
 * needed.  Errors: as the call's shape checks.  Host only. */
bi_status bi_decode_attention_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t max_seq_len,
                                              int64_t split_size, size_t* bytes);

/* One decode step of attention: for request b (one query token) and query
 * head h,  out[b,h,:] = sum_p w_p v_p,  w = softmax_p(scale * q[b,h,:] . k_p)
 * over the request's positions p < seq_lens[b], with k_p, v_p the key/value
 * head h / (Hq / Hkv) (grouped-query attention).
 *   q         [B, Hq, D] bf16, D = 128
 *   k_cache,
 *   v_cache   [num_pages, page_size, Hkv, D] bf16; position p of request b is
 *             row p % page_size of page block_table[b * bt_stride + p / page_size]
 *   block_table [B, bt_stride] int32, seq_lens [B] int32 (device memory)
 *   out       [B, Hq, D] bf16
 * The tree: positions split at multiples of split_size; one warp runs a
 * split over chunks of 16 positions in ascending order with a running (max,
 * sum, output) state in fp32 (scores on the tensor cores with fp32
 * accumulation, exp2 of the log2-scaled scores, weights rounded to bf16
 * before they multiply v and before they are summed); the splits' states
 * fold in split order; out = bf16_rne(o / l).  It depends on seq_lens[b],
 * split_size and D only: no other request, batch size or page placement
 * reaches it, and which warp runs a split, or when, is scheduling only.  An empty request (length 0) gives zeros;
 * NaN / +Inf scores give NaN.
 * Requirements: D == 128; Hq % Hkv == 0 and Hq / Hkv <= 16; page_size a power
 * of two >= 8 with num_pages * page_size < 2^31; split_size a multiple of 64,
 * at most BI_ATTN_MAX_SPLIT (0 = BI_ATTN_DEFAULT_SPLIT); every seq_lens[b] <=
 * max_seq_len <= bt_stride * page_size; B, Hkv and ceil(max_seq_len /
 * split_size) <= 65535 and their product < 2^31; q, caches, out and
 * ws 16-byte aligned, block_table and seq_lens 4-byte aligned; ws_bytes at
 * least bi_decode_attention_workspace_bytes(...).  Cache rows past a
 * request's length are never used (they may hold anything).
 * Device-side checks: a length outside [0, max_seq_len] or a page id outside
 * [0, num_pages) sets BI_ERR_INVALID_ARG in the status that
 * bi_last_device_status() reports; that request's output is then
 * unspecified (NaN for a bad length).
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_ALIGNMENT, BI_ERR_UNSUPPORTED_SHAPE,
 * BI_ERR_WORKSPACE, BI_ERR_CUDA. */
bi_status bi_decode_attention_bf16(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                                   void* out, int64_t B, int64_t Hq, int64_t Hkv, int64_t D,
                                   int64_t num_pages, int64_t page_size, int64_t max_seq_len,
                                   int64_t split_size, float scale, void* ws, size_t ws_bytes,
                                   bi_stream_t stream);

/* Log-probabilities of rows of logits (the lm_head output X [M,V] bf16):
 *   Y[m,v] = x[m,v] - lse_m,  lse_m = max_v x[m,v] + log(sum_v exp(x[m,v] - max)),
 * in fp32, Y [M,V] fp32.  A cluster of 8 CTAs of 512 threads per row: thread
 * g of the cluster folds its 16-byte vectors g, g + 4096, ... in ascending
 * order into a running (max, sum of exp) pair, and the pairs combine by fixed
 * xor butterflies within warps, across warps and across the 8 CTAs (through
 * distributed shared memory), so the tree depends on V only.  expf / logf are CUDA's.  A row holding a NaN or a
 * +Inf, or -Inf everywhere, gives NaN everywhere; otherwise a -Inf logit gives
 * -Inf.
 * Defines: Detent (Batch-Invariant LLM Serving and RL Rollouts at Near-Stock
 * Speed), Sec. 8, Table 6, and CoRun, Sec. IV: per-token log-probabilities
 * are what batch invariance is checked on.  The formula is the textbook one
 * (the pages give none).
 * Requirements: V % 8 == 0, V < 2^31, M < 2^31, X and Y 16-byte aligned; X
 * and Y must not overlap.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_ALIGNMENT, BI_ERR_UNSUPPORTED_SHAPE,
 * BI_ERR_CUDA. */
bi_status bi_log_softmax_bf16(const void* X, float* Y, int64_t M, int64_t V, bi_stream_t stream);

/* out[m] = log-probability of token ids[m] in row m of X [M,V] bf16: the same
 * bits as Y[m, ids[m]] of bi_log_softmax_bf16 (the same kernel arithmetic,
 * without writing the other V - 1 values).  ids: int32 [M] in device memory;
 * an id outside [0, V) gives NaN.  out: fp32 [M].  Requirements and errors as
 * bi_log_softmax_bf16 (ids and out need 4-byte alignment). */
bi_status bi_token_logprobs_bf16(const void* X, const int32_t* ids, float* out, int64_t M, int64_t V,
                                 bi_stream_t stream);

/* Synchronises `stream`, then returns and clears the current device's status
 * word, which holds the first problem a kernel recorded since the last call:
 * BI_OK if none; BI_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out;
 * BI_ERR_INVALID_ARG if decode attention found a device-resident argument
 * (a length or a page id) out of range.  The affected call's output is
 * unspecified.  BI_ERR_CUDA if the synchronisation itself failed. */
bi_status bi_last_device_status(bi_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BI_GEMM_H */
