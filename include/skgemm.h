/*
 * skgemm.h -- C ABI of libskgemm.so: a single-GPU GB300 (sm_103a) GEMM
 *
 *     C = alpha * A * B + beta * C
 *
 * with fp16 / bf16 inputs, fp32 accumulation, a Stream-K work decomposition
 * over persistent CTAs and an optional online ABFT row/column checksum check
 * fused into the epilogue.
 *
 * Sources of the operations (page title, then section / algorithm / figure):
 *  - GEMM definition and shapes: "Stream-K: Work-centric Parallel
 *    Decomposition for Dense Matrix-Matrix Multiplication on the GPU", §A3
 *    (Background). A is m x k, B is k x n, C is m x n, m*n*k MACs.
 *  - Work decomposition: same page, Algorithm 5 (§4, Stream-K), Algorithm 2
 *    (§3.2, data-parallel) and the hybrids of §5.2.
 *  - Partial-tile fixup: same page, Algorithm 5 (StorePartials / Signal /
 *    Wait / LoadPartials) and §4 (the CTA that runs a tile's first
 *    k-iteration writes the tile; here, without ABFT, a tile that eight or
 *    more covering CTAs end in is written in slices by those CTAs).
 *  - ABFT: "Anatomy of High-Performance GEMM with Online Fault Tolerance on
 *    GPUs", thread-level FT-GEMM (Fig. 3: checksums C^c = e^T A B and
 *    C^r = A B e, locate by the mismatching row and column, correct from the
 *    checksum offset) and threadblock-level FT-GEMM (Figs. 5-7: one check per
 *    output tile, checksums updated at every k step).
 *
 * Conventions for every entry point:
 *  - Device pointers are plain CUDA device addresses owned by the caller.
 *    The library allocates no device memory on the gemm path; it reads and
 *    writes only the buffers passed in.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls that
 *    launch work are asynchronous on it.
 *  - Argument errors are returned synchronously and nothing is launched.
 *    Outcomes decided on the device (fixup or pipeline timeouts, ABFT
 *    corrections) are recorded in the workspace report and read back with
 *    skg_report_read after the stream has run the launch.
 *  - No entry point falls back to a CPU path. Unsupported shapes, layouts
 *    or alignments return SKG_ERR_UNSUPPORTED.
 */
#ifndef SKGEMM_H
#define SKGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Input element type of A and B (both the same). */
typedef enum { SKG_IN_F16 = 0, SKG_IN_BF16 = 1 } skg_in_t;

/* Element type of C (and of C0 when beta != 0). */
typedef enum { SKG_OUT_F32 = 0, SKG_OUT_F16 = 1, SKG_OUT_BF16 = 2 } skg_out_t;

/* Storage of A (Stream-K page, problem statement: C = alpha A B + beta C
 * with m, n, k and leading dimensions):
 *   SKG_A_ROW  row-major m x k, element (i,l) at A[i*lda + l], lda >= k:
 *              the "K-major" order the tensor cores read directly;
 *   SKG_A_COL  column-major, element (i,l) at A[l*lda + i], lda >= m
 *              ("M-major"). */
typedef enum { SKG_A_ROW = 0, SKG_A_COL = 1 } skg_a_layout_t;

/* Storage of B:
 *   SKG_B_KMAJOR  stored n x k, element (l,j) at B[j*ldb + l], ldb >= k (the
 *                 "NT" form, as for a weight matrix of a linear layer);
 *   SKG_B_NMAJOR  stored k x n, element (l,j) at B[l*ldb + j], ldb >= n (the
 *                 plain row-major "NN" form).
 * The MMAs read an MN-major operand in place (TMA boxes of 64 MN elements x
 * 64 k, MN-major shared-memory operand descriptors), in the output tiles and
 * in the ABFT checksum GEMMs, and the ABFT encode pass sums its stored rows
 * directly. Only the in-CTA ABFT references (skg_opts_t.abft_local = 2),
 * whose epilogue warps read the stages as K-major rows, run on a K-major
 * copy that a data-movement kernel writes at the end of the workspace (one
 * extra read and write of that operand); size the workspace with
 * skg_workspace_size_layout. */
typedef enum { SKG_B_KMAJOR = 0, SKG_B_NMAJOR = 1 } skg_b_layout_t;

/* Schedules (Stream-K page, §3.2, §4, §5.2):
 *  DP       one persistent CTA walks tiles x, x+g, ... (Algorithm 2 folded
 *           onto g persistent CTAs);
 *  SK       basic Stream-K: all MAC iterations split evenly over g CTAs
 *           (Algorithm 5, even split to within one iteration);
 *  DP_SK1   "data-parallel + one-tile Stream-K": full DP waves, then the
 *           remaining t mod g tiles iteration-balanced over g CTAs;
 *  SK2_DP   "two-tile Stream-K + data-parallel": gives up one DP wave so
 *           each Stream-K CTA gets between one and two tiles of iterations
 *           (the default; the configuration the page evaluates). */
typedef enum {
  SKG_SCHED_DP = 0,
  SKG_SCHED_SK = 1,
  SKG_SCHED_DP_SK1 = 2,
  SKG_SCHED_SK2_DP = 3,
  SKG_SCHED_AUTO = 4  /* chosen per shape by the grid-size model (Stream-K page,
                         App. A.1), with BLK_N and g when those are 0 */
} skg_sched_t;

/* Role of one segment of a CTA's work (Algorithm 5, tile_started /
 * tile_ended): FULL = the CTA computes and stores the whole tile; OWNER =
 * it starts the tile, waits for its peers' partial sums, adds them and
 * stores; PEER = it stores its partial sums to the workspace and signals. */
typedef enum { SKG_ROLE_FULL = 0, SKG_ROLE_OWNER = 1, SKG_ROLE_PEER = 2 } skg_role_t;

typedef enum {
  SKG_OK = 0,
  SKG_ERR_ARG = 1,              /* bad argument (negative size, null pointer, ld too small) */
  SKG_ERR_UNSUPPORTED = 2,      /* valid BLAS call this build does not run (alignment, layout) */
  SKG_ERR_CUDA = 3,             /* a CUDA runtime / driver call failed */
  SKG_ERR_WORKSPACE = 4,        /* workspace missing, misaligned or too small */
  SKG_ERR_FIXUP_TIMEOUT = 5,    /* device: an owner gave up waiting for a peer's partials */
  SKG_ERR_PIPELINE_TIMEOUT = 6, /* device: an internal pipeline wait ran out (never expected) */
  SKG_ABFT_CORRECTED = 16,      /* device: a single fault was located and corrected */
  SKG_ABFT_UNCORRECTABLE = 17   /* device: a checksum mismatch could not be corrected */
} skg_status_t;

/* Largest tile side the library uses (BLK_M = 128, BLK_N <= 256). */
#define SKG_BLK_M 128
#define SKG_BLK_K 64
/* Segments recorded per CTA when a trace buffer is passed. */
#define SKG_TRACE_CAP 255
/* ints per CTA in a trace buffer: 1 count + SKG_TRACE_CAP * 4. */
#define SKG_TRACE_STRIDE 1024
/* Fault records kept in the workspace report. */
#define SKG_MAX_RECORDS 64

/* Options of one gemm call. Zero-initialised fields select the defaults;
 * call skg_opts_default to get them explicitly. */
typedef struct {
  int32_t sched;        /* skg_sched_t (default SKG_SCHED_AUTO) */
  int32_t grid;         /* g, persistent CTAs; 0 = chosen by the model (AUTO)
                           or the number of SMs (fixed schedule). At most the
                           number of SMs: all CTAs must be co-resident, since
                           a tile owner waits for later CTAs. */
  int32_t tile_n;       /* BLK_N: 64, 128 or 256; 0 = chosen by the model.
                           64 (the small-tile configuration: 128 x 64 tiles,
                           half the operand bytes per MAC iteration and per
                           partial tile) is for GEMMs without ABFT on single
                           CTAs: with abft or cta_pair = 2 it returns
                           SKG_ERR_UNSUPPORTED, and the model picks it by
                           itself only for those GEMMs. */
  int32_t abft;         /* 0 = off; 1 = verify every output tile, locate and
                           correct a single fault, report the rest */
  float tau_row;        /* ABFT row threshold; <= 0 = the default
                           2^-12 * sqrt(k) * sqrt(BLK_N) * max|A| * max|B| */
  float tau_col;        /* ABFT column threshold; <= 0 = the default
                           2^-12 * sqrt(k) * sqrt(BLK_M) * max|A| * max|B| */
  int32_t inject_tile;  /* fault injection for testing: < 0 = none; else the
                           tile index whose accumulator gets one bit flipped */
  int32_t inject_row;   /* row within the tile [0, 128) */
  int32_t inject_col;   /* column within the tile [0, BLK_N) */
  int32_t inject_bit;   /* bit of the fp32 accumulator [0, 32) */
  uint64_t timeout_ns;  /* bound on every device-side wait; 0 = 2 s */
  int32_t* trace;       /* optional device buffer, grid * SKG_TRACE_STRIDE
                           int32: per CTA the segment count, then
                           (tile, k_iter_begin, k_iter_end, role) per segment */
  uint64_t* cta_clock;  /* optional device buffer, grid * 2 uint64: per CTA
                           the %globaltimer at start and end (ns) */
  int32_t test_drop_signal; /* testing only: 1 + index of a CTA that skips its
                           Stream-K Signal, so the owner's bounded wait runs out
                           and the launch reports SKG_ERR_FIXUP_TIMEOUT; 0 = none */
  int32_t abft_preencoded; /* 1 = skg_abft_encode already wrote the encodings
                           of this call's A and B (same shape and options) into
                           the workspace, so skg_gemm skips the encode pass and
                           only forms the checksums from them */
  int32_t raster_band;  /* output tiles are visited in bands of this many tile
                           columns, row by row inside a band (L2 reuse);
                           0 = chosen by the library; >= the number of tile
                           columns = plain row-major order */
  int32_t cta_pair;     /* 0 = the library decides (pairs when their 256 x 256
                           tiles fill every resident cluster and neither grid
                           nor BLK_N 128 is requested),
                           1 = single CTAs, 2 = clusters of two CTAs that run
                           256 x 256 tiles with one M = 256 tcgen05 MMA (each
                           CTA loads its 128 rows of A and half of B per
                           k-step); requires BLK_N 256, and with ABFT the
                           checksum GEMMs then run as separate launches.
                           `grid` counts CTAs and must then be even. */
  int32_t abft_local;   /* ABFT reference checksums formed inside each CTA
                           from the operand tiles in shared memory while the
                           MMAs run ("Anatomy of High-Performance GEMM with
                           Online Fault Tolerance on GPUs", threadblock-level
                           FT-GEMM): no encode pass and no checksum GEMMs, for
                           a data-parallel plan of at most one 128 x 128
                           output tile per SM on single CTAs. The CUDA-core
                           sums take several times the MMAs' time per k-step
                           on GB300, so 0 (default) and 1 = never, 2 =
                           whenever the shape allows it. */
  int32_t inject2_tile; /* a second injected flip for testing, in the same
                           form as inject_*: < 0 = none. Two flips in one
                           tile make the mismatch pattern the single-fault
                           rule cannot correct; in two tiles, two corrections */
  int32_t inject2_row;
  int32_t inject2_col;
  int32_t inject2_bit;
  int32_t inject_kstep; /* < 0 (default): the inject_* flip is applied to the
                           fixed-up accumulator just before the check. >= 0:
                           it is applied inside the mainloop instead, in TMEM,
                           right after the MMAs of the tile's MAC iteration
                           inject_kstep (0 <= inject_kstep < ceil(k / 64)),
                           to the partial accumulator of the CTA that runs
                           that iteration; later iterations and the Stream-K
                           fixup then add onto the faulty value. inject2_* is
                           always applied before the check. */
  int32_t stagger;      /* StaggerU-style k-offset staggering: 0 or 1 = off;
                           s > 1 = CTA x starts each of its work items at
                           MAC iteration ((x mod s) * n) / s of the item's n
                           iterations and wraps around to its first one, so
                           CTAs that read the same operand columns do not all
                           start at the same k. Sums are re-associated only. */
  int32_t abft_inloop;  /* ABFT reference checksums accumulated inside the
                           mainloop: every k-step also runs the checksum MMAs
                           cr += A_s (B e)_s and cc += B_s (e^T A)_s on the
                           stage's operand tiles and the encodings of that
                           k-step, into TMEM next to the accumulator, so no
                           separate checksum tiles run and no verification
                           waits for other CTAs. Data-parallel plans of
                           128 x 128 tiles or 256 x 256 CTA-pair tiles,
                           K-major operands. 0 = the library decides,
                           1 = never, 2 = whenever the call allows it. */
} skg_opts_t;

/* One segment of a schedule (Stream-K page, Algorithm 5 / §5.2). k_iter_*
 * count MAC iterations of BLK_K within the tile. */
typedef struct {
  int32_t cta;
  int32_t tile;         /* tile index; with raster_band >= tiles_n it is
                           row-major, tile = tm * tiles_n + tn */
  int32_t k_iter_begin;
  int32_t k_iter_end;   /* exclusive */
  int32_t role;         /* skg_role_t */
} skg_segment_t;

/* One located (or uncorrectable) checksum mismatch. */
typedef struct {
  uint32_t launch;      /* launch epoch of the workspace (1 for the first launch) */
  int32_t tile;
  int32_t row;          /* row within the tile, -1 if not located */
  int32_t col;          /* column within the tile, -1 if not located */
  int32_t status;       /* SKG_ABFT_CORRECTED or SKG_ABFT_UNCORRECTABLE */
  int32_t n_bad_rows;
  int32_t n_bad_cols;
  uint32_t injected;    /* 1 if the flip came from skg_opts_t.inject_* */
  float before;         /* accumulator value as checked (the faulty one) */
  float after;          /* value written back after correction */
  float delta_row;      /* row checksum mismatch at the located row */
  float delta_col;      /* column checksum mismatch at the located column */
  float clean_value;    /* for injected flips: the value before the flip */
  uint32_t pad[3];
} skg_fault_record_t;

/* Device-side outcome counters, cumulative over launches on one workspace
 * until read with reset != 0. */
typedef struct {
  uint32_t status_bits;   /* bit (1 << code) set for each device outcome code seen */
  uint32_t launches;      /* launches that ran to completion */
  uint32_t tiles_checked; /* output tiles verified by ABFT */
  uint32_t detected;      /* tiles with at least one checksum mismatch */
  uint32_t corrected;
  uint32_t uncorrectable;
  uint32_t timeouts;      /* device waits that ran out */
  uint32_t n_records;     /* records written (at most SKG_MAX_RECORDS kept) */
  float max_ratio_row;    /* largest |row mismatch| / tau_row over rows that passed */
  float max_ratio_col;    /* same for columns */
  float tau_row;          /* largest thresholds used by the ABFT launches */
  float tau_col;
  uint32_t mid_injected;  /* mid-mainloop flips applied (skg_opts_t.inject_kstep) */
  float mid_before;       /* the partial accumulator value the latest one flipped */
  float mid_after;        /* and the value it left in TMEM */
  uint32_t reserved;
  skg_fault_record_t records[SKG_MAX_RECORDS];
} skg_report_t;

/* Fill *opts with the defaults (schedule, g and BLK_N chosen by the model,
 * ABFT off, no injection, 2 s wait bound, no trace). */
void skg_opts_default(skg_opts_t* opts);

/* Bytes of device workspace a gemm of this shape needs with these options
 * (opts may be NULL): a header with the launch epoch and the report, one
 * flag and one fp32 BLK_M x BLK_N partial-sum slot per CTA (Stream-K page,
 * §4: fixup storage scales with g, not with the problem), the partial
 * checksums, and with ABFT the split encodings e^T A and B e. Two banks of
 * flags and slots: with ABFT the second serves the fused checksum tiles;
 * without, the split reduction (a Stream-K tile that two or more of its
 * CTAs end their ranges in is finished by those CTAs together, each storing
 * a range of its columns), whose owners keep their partial there when they
 * already hold one of an earlier tile. */
size_t skg_workspace_size(int64_t m, int64_t n, int64_t k, const skg_opts_t* opts);

/* skg_workspace_size for the given operand layouts: when opts select the
 * in-CTA ABFT references, the same bytes plus room for the K-major copies of
 * MN-major operands (m x k and n x k elements, rows rounded up to 16 bytes);
 * otherwise equal to skg_workspace_size. 0 for an unknown layout or invalid
 * arguments. */
size_t skg_workspace_size_layout(int64_t m, int64_t n, int64_t k, int32_t a_layout,
                                 int32_t b_layout, const skg_opts_t* opts);

/* Zero a workspace (`bytes` from skg_workspace_size) before its first use.
 * Afterwards the library keeps it consistent itself, also when the same
 * workspace serves calls of other shapes and options (large enough for each):
 * the header, report and flags sit at fixed offsets and the flags carry a
 * launch epoch, so they never need clearing, and every other region is
 * written by a call before that call reads it. Asynchronous on `stream`. */
skg_status_t skg_workspace_init(void* workspace, size_t bytes, void* stream);

/* C = alpha * A B + beta * C, asynchronous on `stream`.
 *   A: device, in_dtype, stored as a_layout says (skg_a_layout_t), lda in
 *      elements (>= k row-major, >= m column-major).
 *   B: device, in_dtype, stored as b_layout says (skg_b_layout_t), ldb
 *      >= k (K-major) or >= n (N-major).
 *   C: device, out_dtype, row-major m x n, ldc >= n; read only if beta != 0.
 *   A, B, C must be 16-byte aligned and lda, ldb, ldc must be multiples of
 *   16 bytes (the TMA engine's rule); otherwise SKG_ERR_UNSUPPORTED. An
 *   unknown layout value or a leading dimension below its minimum is
 *   SKG_ERR_ARG.
 *   workspace: device, >= skg_workspace_size_layout(m, n, k, a_layout,
 *   b_layout, opts) bytes (skg_workspace_size for K-major operands), zeroed
 *   once with skg_workspace_init; one workspace per stream (two launches
 *   that share a workspace must not overlap).
 *   opts: NULL for defaults. m, n or k of zero is valid (k = 0 gives
 *   C = beta * C). */
skg_status_t skg_gemm(int64_t m, int64_t n, int64_t k, float alpha, const void* A, int64_t lda,
                      const void* B, int64_t ldb, float beta, void* C, int64_t ldc,
                      int32_t in_dtype, int32_t out_dtype, int32_t a_layout, int32_t b_layout,
                      const skg_opts_t* opts, void* workspace, size_t ws_bytes, void* stream);

/* skg_gemm with the checksum check forced on (opts->abft = 1): every output
 * tile's fp32 accumulator A_tile B_tile is verified against the reference
 * checksums (e^T A) B and A (B e) before alpha, beta and the cast are
 * applied; a single fault is located and corrected, anything else is
 * reported. Results land in the workspace report (skg_report_read). */
skg_status_t skg_gemm_verify(int64_t m, int64_t n, int64_t k, float alpha, const void* A,
                             int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                             int64_t ldc, int32_t in_dtype, int32_t out_dtype, int32_t a_layout,
                             int32_t b_layout, const skg_opts_t* opts, void* workspace,
                             size_t ws_bytes, void* stream);

/* The ABFT encode pass of skg_gemm_verify on its own (one kernel): e^T A
 * over each 128-row tile of A and B e over each BLK_N-column tile of B,
 * each split into hi and lo terms of the input type with a per-tile scale,
 * plus per-tile max |A| and max |B| for the default thresholds ("Anatomy of
 * High-Performance GEMM with Online Fault Tolerance on GPUs",
 * threadblock-level ABFT, Fig. 5: the encodings e^T A and B e of each
 * threadblock's operands). Arguments as for skg_gemm with K-major operands
 * (A row-major, B stored n x k; skg_abft_encode_layout takes the layouts);
 * opts must be the options of the gemm call that follows with
 * opts->abft_preencoded = 1. Asynchronous on `stream`. */
skg_status_t skg_abft_encode(int64_t m, int64_t n, int64_t k, const void* A, int64_t lda,
                             const void* B, int64_t ldb, int32_t in_dtype,
                             const skg_opts_t* opts, void* workspace, size_t ws_bytes,
                             void* stream);

/* skg_abft_encode for operands in any layout (skg_a_layout_t,
 * skg_b_layout_t): an MN-major operand's encodings are the sums of its
 * stored row segments. For a following pre-encoded call with the same
 * layouts (which then reads MN-major operands in place). */
skg_status_t skg_abft_encode_layout(int64_t m, int64_t n, int64_t k, const void* A, int64_t lda,
                                    const void* B, int64_t ldb, int32_t in_dtype,
                                    int32_t a_layout, int32_t b_layout, const skg_opts_t* opts,
                                    void* workspace, size_t ws_bytes, void* stream);

/* The schedule the kernel runs, computed on the host: for every CTA, its
 * ordered segments (tile, k-iteration range, role). bm, bn, bk are the tile
 * sides (bn = the BLK_N skg_gemm would use; pass skg_tile_n to get it).
 * Writes at most `cap` segments to `out` (host memory, may be NULL when
 * cap == 0) and the total count to *n_out. */
skg_status_t skg_schedule_query(int64_t m, int64_t n, int64_t k, int32_t bm, int32_t bn,
                                int32_t bk, int32_t g, int32_t sched, skg_segment_t* out,
                                int64_t cap, int64_t* n_out);

/* Predicted run time (microseconds) of one launch with this schedule under
 * the library's grid-size model (Stream-K page, App. A.1: the slowest CTA's
 * fixed cost + per-iteration cost + partial-store cost + per-peer cost, with
 * constants fitted on GB300). bm must be 128 and bn 64, 128 or 256. */
skg_status_t skg_schedule_cost(int64_t m, int64_t n, int64_t k, int32_t bm, int32_t bn,
                               int32_t bk, int32_t g, int32_t sched, double* us);

/* BLK_N, grid g and schedule skg_gemm would use for this shape and options
 * (the model's choice for whatever opts leaves open). Any out pointer may be
 * NULL. */
skg_status_t skg_launch_shape(int64_t m, int64_t n, int64_t k, const skg_opts_t* opts,
                              int32_t* tile_n, int32_t* grid, int32_t* sched);

/* The launch plan skg_gemm would use for this shape and options. */
typedef struct {
  int32_t tile_m;      /* output rows per tile: 128, or 256 for CTA pairs */
  int32_t tile_n;      /* BLK_N: 64, 128 or 256 */
  int32_t ctas;        /* CTAs launched for the output tiles */
  int32_t cta_pair;    /* 1 = single CTAs, 2 = clusters of two CTAs */
  int32_t sched;       /* skg_sched_t */
  int32_t side_ctas;   /* extra CTAs for the ABFT checksum tiles (0 =
                          checksum tiles split over the CTAs above) */
  int32_t fused_checksums; /* ABFT: 1 = checksum GEMMs run inside the main
                          launch, 0 = as separate launches (or no ABFT) */
  int32_t encode_in_kernel; /* ABFT: 1 = the side CTAs also run the encode
                          pass, so the call is a single launch */
  int32_t local_checksums; /* ABFT: 1 = the reference checksums are formed in
                          each CTA (skg_opts_t.abft_local), a single launch */
  int32_t inloop_checksums; /* ABFT: 1 = the reference checksums are
                          accumulated by the output tiles' MMAs
                          (skg_opts_t.abft_inloop), after the encode pass */
  int32_t side_checksum_ctas; /* of the side CTAs, the first this many run the
                          checksum tiles (split evenly over them); the others
                          only take part in the in-kernel encode pass */
} skg_plan_t;

/* Same choice as skg_launch_shape, with the CTA-pair and checksum-tile
 * placement. Both queries plan for bf16 inputs: for fp16 with ABFT the
 * encode pass is always a separate launch and the side CTAs are only the
 * checksum tiles' (one per tile). */
skg_status_t skg_launch_plan(int64_t m, int64_t n, int64_t k, const skg_opts_t* opts,
                             skg_plan_t* out);

/* Copy the workspace report to host memory (synchronises `stream` first);
 * reset != 0 also clears the counters and records. */
skg_status_t skg_report_read(const void* workspace, skg_report_t* out, int32_t reset,
                             void* stream);

/* Size of the fixed device scratch array behind skg_gemm_noalloc. */
#define SKG_NOALLOC_SCRATCH_BYTES (16u << 20)

/* skg_gemm without a caller workspace, for callers that cannot allocate
 * device memory (for example a plugin whose host framework owns all device
 * memory through its own allocator, or a latency-critical path that cannot
 * afford cudaMalloc's implicit synchronisation). The pages have no
 * counterpart: this is a packaging choice of this library. The Stream-K
 * workspace comes from one file-scope device array of
 * SKG_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU loading the library
 * holds until exit; nothing is allocated per call. The first call on a
 * device sets that device up (looks up the array's address and clears its
 * header, report and flags on `stream`), so make it before any stream
 * capture. All calls share the array and it keeps the last call's contents;
 * calls of different shapes and options may follow each other, but calls
 * whose launches overlap on the GPU race and must not be issued. BLK_N
 * defaults to 128 here (unless opts asks for CTA pairs). A shape or option
 * set whose workspace exceeds the array returns SKG_ERR_WORKSPACE: on a
 * 152-SM GB300 that is every ABFT call with opts->grid = 0 (its checksum
 * GEMMs may use every SM, about 40 MB of partial slots); ABFT with a small
 * explicit grid fits. Device-side outcomes are read with
 * skg_noalloc_report_read. Other arguments and errors as for skg_gemm. */
skg_status_t skg_gemm_noalloc(int64_t m, int64_t n, int64_t k, float alpha, const void* A,
                              int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                              int64_t ldc, int32_t in_dtype, int32_t out_dtype, int32_t a_layout,
                              int32_t b_layout, const skg_opts_t* opts, void* stream);

/* skg_report_read for the current device's skg_gemm_noalloc array: copies
 * its report (timeouts, ABFT detections and corrections of every noalloc
 * call since the last reset) to host memory after synchronising `stream`;
 * reset != 0 also clears it. Sets the device up like skg_gemm_noalloc's
 * first call when that has not happened yet. */
skg_status_t skg_noalloc_report_read(skg_report_t* out, int32_t reset, void* stream);

/* Bytes of device staging memory skg_gemm_host needs for this problem:
 * packed device copies of A and B as stored (rows rounded up to 16 bytes)
 * and of C (m rows of n outputs, rounded up to 16 bytes). 0 for invalid
 * arguments. */
size_t skg_host_staging_size(int64_t m, int64_t n, int64_t k, int32_t in_dtype,
                             int32_t out_dtype, int32_t a_layout, int32_t b_layout);

/* skg_gemm on operands in HOST memory, asynchronous on `stream`: copies A
 * and B (and C when beta != 0) into `staging` (device memory, >=
 * skg_host_staging_size bytes, caller-owned), runs skg_gemm (or
 * skg_gemm_verify when opts->abft = 1) on the device copies, and copies C
 * back to the host. A, B, C are host pointers with the meanings of
 * skg_gemm (any alignment; leading dimensions in elements); page-locked
 * host memory lets the copies run asynchronously and overlap with work on
 * other streams. workspace as for skg_gemm with these layouts
 * (skg_workspace_size_layout). Copies are one cudaMemcpy2DAsync per matrix.
 * The host buffers must stay valid, and C unread, until `stream` has
 * reached this point. */
skg_status_t skg_gemm_host(int64_t m, int64_t n, int64_t k, float alpha, const void* A,
                           int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                           int64_t ldc, int32_t in_dtype, int32_t out_dtype, int32_t a_layout,
                           int32_t b_layout, const skg_opts_t* opts, void* staging,
                           size_t staging_bytes, void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace skg_gemm_f64 needs: a header (launch epoch,
 * exit tickets), the report, one flag and one 64 x 64 fp64 partial-tile slot
 * per CTA (Stream-K page, §4: fixup storage scales with g). */
size_t skg_workspace_size_f64(int64_t m, int64_t n, int64_t k, const skg_opts_t* opts);

/* fp64 Stream-K GEMM (Stream-K page, §6 evaluates FP64 as well as FP16):
 * C = alpha * A B + beta * C, all double, asynchronous on `stream`. A
 * row-major m x k (lda >= k), B stored n x k (ldb >= k), C row-major m x n
 * (ldc >= n), device pointers, leading dimensions in elements. The MAC
 * iterations of 64 x 64 x 16 tiles are split over opts->grid persistent CTAs
 * (0 = one per SM) with opts->sched (SKG_SCHED_AUTO = the two-tile hybrid),
 * partial tiles fixed up through the workspace with epoch flags as in
 * skg_gemm; CUDA-core FMAs (GB300's fp64 rate is far below its 16-bit
 * tensor rate). workspace: device, 256-byte aligned, >=
 * skg_workspace_size_f64 bytes, zeroed once with skg_workspace_init; one
 * per stream. A fixup wait that runs out is reported as
 * SKG_ERR_FIXUP_TIMEOUT in the report (skg_report_read). k = 0 gives
 * C = beta * C. No ABFT in this variant. */
skg_status_t skg_gemm_f64(int64_t m, int64_t n, int64_t k, double alpha, const double* A,
                          int64_t lda, const double* B, int64_t ldb, double beta, double* C,
                          int64_t ldc, const skg_opts_t* opts, void* workspace, size_t ws_bytes,
                          void* stream);

/* Number of SMs of the current device (0 if there is no device). */
int32_t skg_device_sm_count(void);

/* Short text for a status code. */
const char* skg_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* SKGEMM_H */
