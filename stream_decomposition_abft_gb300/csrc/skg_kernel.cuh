// Persistent Stream-K GEMM kernel for sm_103a with an optional fused ABFT
// check.
//
//   C = alpha * A B + beta * C,   A: m x k (K-major), B: stored n x k (K-major)
//
// (Either operand may also be MN-major -- A stored k x m, B stored k x n:
// the producer then loads 64 x 64-element boxes and the MMAs read MN-major
// shared-memory operands, in output and checksum tiles alike; see
// KernelParams::a_mn.)
//
// Work decomposition: "Stream-K: Work-centric Parallel Decomposition for
// Dense Matrix-Matrix Multiplication on the GPU", Algorithm 5 and §5.2
// (see skg_sched.cuh). One CTA per SM walks its segments:
//
//   warp 0      TMA producer: A and B tiles (BLK_K = 64, 128-byte swizzle)
//               into a STAGES-deep shared-memory ring, full/empty mbarriers.
//   warp 1      MMA issuer: tcgen05.mma kind::f16, M = 128, N = BLK_N, fp32
//               accumulator in TMEM (double-buffered when it fits), commit
//               to the ring's empty barrier and to the accumulator barrier.
//   warps 2-5   epilogue (TMEM lane quadrant = warp % 4, one output row per
//               thread): a PEER segment writes its fp32 partial tile to the
//               workspace and releases a flag carrying the launch epoch
//               (StorePartials / Signal); an OWNER waits for its later peers'
//               flags and adds their partials (Wait / LoadPartials), pulled
//               through the idle stage ring with bulk copies since an owned
//               tile is always its CTA's last work; then alpha / beta, the
//               output cast, a swizzled staging buffer and a TMA store
//               (StoreTile). The tile's k = 0 CTA writes C (§4), except that
//               without ABFT a tile split over eight or more CTAs that all
//               end in it is reduced and written in slices by all of them
//               (reduce_share); either way C needs no atomics.
//
// ABFT ("Anatomy of High-Performance GEMM with Online Fault Tolerance on
// GPUs", Figs. 3 and 5-7): an encode pass (its own launch, or the first work
// of dedicated side CTAs) forms e^T A per 128-row tile and B e per
// BLK_N-column tile; two skinny tensor-core GEMMs, run as the first tiles of
// this same launch (side tiles), form the reference checksums
// cr = A (B e) and cc = (e^T A) B of every output tile. The
// epilogue of each tile's owner, after the Stream-K fixup, forms the row sums
// (in-thread) and column sums (warp transpose-reduction + shared memory) of
// the fp32 accumulator, compares them with cr and cc, locates a single fault
// at the mismatching row and column, replaces it by
// cr[i*] - sum_{j != j*} acc[i*, j], and only then applies alpha / beta and
// stores. The checksums never pass through the mainloop, so the MMA reads
// each operand tile from shared memory once (a separate N = 16 checksum MMA
// would read the whole A or B tile again and halve the tensor-core rate on
// shared-memory bandwidth).
//
// Every wait (mbarrier or peer flag) is bounded by a %globaltimer deadline;
// on expiry the kernel records the error in the workspace report, sets a
// CTA-wide abort flag, drains its own copies and MMAs, frees TMEM and exits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "skg_ptx.cuh"
#include "skg_sched.cuh"
#include "skgemm.h"

namespace skg {

constexpr int kBM = 128;
constexpr int kBK = 64;
// MN-major operand box: 64 MN elements (one 128-byte swizzled row) x kBK.
constexpr int kMnBox = 64;
constexpr int kMnBoxBytes = kMnBox * kBK * 2;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
static_assert(kThreads == 64 + kEpiThreads && kEpiThreads == 128,
              "epi_all and the named barriers count the four epilogue warps");
constexpr int kEncRows = 2;  // hi and lo terms of each encoding
constexpr int kFixSlots = 6;  // per epilogue warp: staged partial pieces in flight
constexpr int kAuxBytes = 1024;  // shared-memory bookkeeping (struct Aux) after the staging
constexpr uint32_t kSmemLimit = 232448;
// Flags per fixup region. The flag array has a fixed place and size in every
// workspace (two regions of kMaxCtas), so a workspace reused for another
// shape or option set never finds other data where its flags now lie; a
// launch uses at most kMaxCtas CTAs.
constexpr int kMaxCtas = 1024;

// Workspace header (device). The report follows at offset 256.
// The epoch is advanced once per launch by the CTA that takes the launch's
// last ticket (every CTA takes one after reading the epoch); a launch that
// read epoch e flags with e + 1 and counts in ck_done[e & 1] / enc_done[e & 1],
// and the last-ticket CTA clears the other parity for the next launch.
struct WsHeader {
  uint32_t epoch;        // launches on this workspace
  uint32_t done;         // CTA tickets of the running launch
  uint32_t ck_done[2];   // fused checksum tiles stored, by epoch parity
  uint32_t enc_done[2];  // side CTAs done with the in-kernel encode pass, by parity
  uint32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// What the ABFT encode pass publishes per operand tile for the main
// kernel's epilogue.
struct TilePub {
  int32_t scale_exp;  // the tile's encodings are stored scaled by 2^scale_exp
  int32_t pad;
};

struct KernelParams {
  Schedule s;
  int m, n, k;
  float alpha, beta;
  uint32_t idesc_main;
  // MN-major operands: A stored k x m and / or B stored k x n, loaded as
  // 64 x 64-element boxes (64 MN elements = one 128-byte swizzled row per k)
  // and read by the MMAs as MN-major shared-memory operands. They also form
  // the A operand of the fused checksum tiles (A for cr, B for cc); the
  // encodings (their B operand) are always K-major.
  int32_t a_mn, b_mn;
  WsHeader* hdr;
  skg_report_t* report;
  // Fixup storage: region 0 (output tiles) uses flags[0, kMaxCtas) and
  // partial slots [0, ws_ctas); region 1 (fused checksum tiles) flags
  // [kMaxCtas, 2 kMaxCtas) and the next ws_ctas slots. Slot x holds
  // kBM x BN fp32 values.
  uint32_t* flags;
  float* partials;
  int ws_ctas;
  // ABFT reference checksums (hi and lo partial products, scaled):
  // row checksums cr_all[row * ld_cr + 2 * tn + t] = A (B e)_tn, and column
  // checksums ccT_all[col * ld_cc + 2 * tm + t] = ((e^T A)_tm B)^T.
  const float* cr_all;
  const float* cc_all;
  int64_t ld_cr, ld_cc;
  const TilePub* pub_a;  // per 128-row tile of A
  const TilePub* pub_b;  // per BLK_N-column tile of B
  // max |element| of every encode unit (operand tile x slice of enc_slices
  // per tile; A tiles first): a tile's maximum is the max over its units.
  const float* umax;
  int enc_slices, enc_tiles_a;
  // In-kernel encode pass (bf16; the separate encode kernel's work, run by
  // the dedicated side CTAs before their checksum tiles): units of one
  // operand tile x 256 k-columns, boxes of 64 rows.
  int enc_inkernel;
  int enc_tiles_b, enc_bn, enc_kp;
  void* enc_a_w;
  void* enc_b_w;
  float* umax_w;
  TilePub* pub_w;
  // Fused reference-checksum GEMMs: tiles [0, s.t_ck) of the schedule.
  // Tile j < ck_cr_tiles computes rows [128 j, 128 j + 128) of
  // cr_all = A x [Be_hi; Be_lo]^T (ck_n_cr columns); the others compute rows
  // of ccT_all = B x [eA_hi; eA_lo]^T (ck_n_cc columns). Both store fp32.
  // With CTA pairs a side tile is two such 128-row tiles (2j for the leader,
  // 2j + 1 for its peer), and each CTA loads half of the encoding rows.
  int ck_cr_tiles;
  int ck_n_cr, ck_n_cc;
  int ck_rows_cr, ck_rows_cc;  // encoding rows loaded per k-step (N rounded up to 16)
  // k-blocks per ring stage for checksum tiles (1 or 2): a checksum k-step
  // needs only the A (or B) tile and a few encoding rows, so two fit in one
  // BLK_N = 256 stage; packed stages hold A(k), A(k+1), enc(k), enc(k+1).
  int ck_kpack_cr, ck_kpack_cc;
  // ck_atomic (with the in-kernel encode pass, whose CTAs zero cr_all and
  // ccT_all before they report): every checksum-tile segment adds its rows
  // into them with a TMA reduce-add, whatever its Stream-K role, so no
  // segment waits for another; ck_target segment reports (kCkHalf per
  // segment) mean all of them landed.
  int ck_atomic;
  int ck_target;
  uint32_t idesc_cr, idesc_cc;
  float tau_row, tau_col;  // <= 0: derive from the encode pass maxima
  // Fault injection (testing only): up to two single-bit flips of the fp32
  // accumulator, slot s at (inj_row[s], inj_col[s]) of 128 x BLK_N output
  // tile inj_tile[s] (< 0: slot unused). inj_kb >= 0 applies slot 0 inside
  // the mainloop, after the tile's MAC iteration inj_kb, instead of after
  // the fixup.
  int inj_tile[2], inj_row[2], inj_col[2], inj_bit[2];
  int inj_kb;
  // StaggerU-style k staggering: > 1 rotates each work item's k order by
  // ((unit mod stagger) * n) / stagger of its n iterations.
  int stagger;
  uint64_t timeout_ns;
  int32_t* trace;
  uint64_t* cta_clock;
  int drop_signal;  // testing: CTA index that skips its Signal, or -1
  int in_f16;       // inputs are fp16 (else bf16): the in-CTA ABFT sums read them
  // C (and C0) for the shared tile reduction's plain stores: ldc elements
  // per row, the output type of the launch.
  void* c_ptr;
  int64_t ldc;
};


__host__ __device__ constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p *= 2;
  return p;
}

template <int BN_, bool ABFT_, int OUT_, bool PAIR_ = false, bool LOCAL_ = false, bool MN_ = false,
          bool ILC_ = false>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr bool ABFT = ABFT_;
  // 64-wide tiles (the small-tile configuration): plain GEMMs on single
  // CTAs; the ABFT column references come in 128-column groups.
  static_assert(BN_ >= 128 || (!ABFT_ && !PAIR_ && !LOCAL_ && !ILC_),
                "64-wide tiles: plain GEMMs on single CTAs");
  // 128-column groups of the tile (ABFT column references; at least one so
  // that the arrays sized by it exist for 64-wide tiles too).
  static constexpr int CC_GROUPS = BN_ >= 128 ? BN_ / 128 : 1;
  // In-loop reference checksums: every k-step also issues the checksum MMAs
  // cr += A_s (B e)_s and cc += B_s (e^T A)_s into TMEM columns next to the
  // accumulator, from encodings the encode pass wrote (loaded with each
  // stage), so no separate checksum tiles run. Data-parallel plans only (no
  // tile is split), K-major operands.
  static constexpr bool ILC = ILC_;
  static_assert(!ILC_ || (ABFT_ && !LOCAL_ && !MN_), "in-loop checksums: ABFT, K-major");
  static_assert(!ILC_ || BN_ == 128 || PAIR_, "in-loop checksums: 128-wide tiles or CTA pairs");
  // MN-major operands possible (KernelParams::a_mn / b_mn); the K-major-only
  // instantiations carry no layout code in the producer and MMA loops.
  static constexpr bool MN = MN_;
  static_assert(!(MN_ && LOCAL_), "in-CTA references read K-major stages");
  // In-CTA ABFT references (local_checksums): the epilogue warps also read
  // every stage, for launches of at most one whole tile per CTA.
  static constexpr bool LOCAL = LOCAL_;
  static_assert(!LOCAL || (ABFT_ && !PAIR_), "in-CTA references need ABFT on single CTAs");
  static constexpr int OUT = OUT_;  // 0 = f32, 1 = f16, 2 = bf16
  // CTA pairs: a cluster of two CTAs runs 256 x BN tiles with one M = 256
  // MMA; each CTA loads its 128 rows of A and BN / 2 rows of B per stage.
  static constexpr bool PAIR = PAIR_;
  static constexpr int OUT_BYTES = OUT == 0 ? 4 : 2;
  static constexpr int EPI_COLS = 128 / OUT_BYTES;  // one 128-byte staging row
  // TMEM columns per accumulator buffer: the tile, then (ILC) 16 columns of
  // row-checksum sums (cr: hi, lo) and 16 of column-checksum sums (cc: hi,
  // lo; for a CTA pair also the other half's at +8).
  static constexpr int CR_COL = BN;
  static constexpr int CC_COL = BN + 16;
  static constexpr int ACC_COLS = BN + (ILC ? 32 : 0);
  static constexpr int ACC_BUFS = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_COLS = pow2_at_least(ACC_BUFS * ACC_COLS);
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // rows of B this CTA loads
  static constexpr int B_BYTES = B_ROWS * kBK * 2;
  // ILC: each stage also holds the k-step's encodings as the N = 16 B operand
  // of the checksum MMAs (rows hi, lo, then zeros; a CTA pair splits N, so
  // each CTA holds 8 rows): e^T A of this CTA's 128 rows, and B e of the tile.
  static constexpr int ENC_ROWS = PAIR ? 8 : 16;
  static constexpr int ENC_SLOT_BYTES = ILC ? ENC_ROWS * 128 : 0;
  static constexpr int ENCA_OFF = A_BYTES + B_BYTES;
  static constexpr int ENCB_OFF = ENCA_OFF + ENC_SLOT_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + 2 * ENC_SLOT_BYTES;
  static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t ENC_BOX_BYTES = 2 * kBK * 2;  // hi and lo rows of one k-step
  // Packed checksum stage: two A tiles, then two encoding slots of ENC_SLOT bytes.
  static constexpr int ENC_SLOT = 8192;
  static constexpr bool CK_PACK = !PAIR && STAGE_BYTES >= 2 * A_BYTES + 2 * ENC_SLOT;
  static constexpr int EPI_BUF_BYTES = 32 * 128;
  static constexpr int EPI_BUFS = 2;
  static constexpr int EPI_BYTES = 4 * EPI_BUFS * EPI_BUF_BYTES;
  static constexpr int AUX_BYTES = kAuxBytes;
  // The ABFT column partial sums of warp q (BN floats) live in warp q's own
  // first staging buffer, which is idle while a tile is being verified.
  static_assert(BN * 4 <= EPI_BUF_BYTES, "column sums must fit one staging buffer");
  // ILC with CTA pairs: each CTA's TMEM holds the column sums of its 128 B
  // rows for both halves' e^T A; the halves swap the other's through this
  // buffer (two tiles' worth, 128 floats each).
  static constexpr int XBUF_BYTES = (ILC && PAIR) ? 2 * 128 * 4 : 0;
  static constexpr int STAGES_FIT =
      (int)((kSmemLimit - 1024 - EPI_BYTES - AUX_BYTES - XBUF_BYTES) / STAGE_BYTES);
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr uint32_t SMEM_BYTES =
      1024 + STAGES * STAGE_BYTES + EPI_BYTES + AUX_BYTES + XBUF_BYTES;
  static_assert(STAGES >= 2, "shared memory too small for two stages");
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory over the per-CTA limit");
  static_assert(TMEM_COLS <= 512, "TMEM over 512 columns");
  static_assert(BN % EPI_COLS == 0, "epilogue chunking");
};

// Shared-memory bookkeeping that lives after the stage ring and staging.
struct Aux {
  uint64_t bars[60];      // full[S], empty[S], tfull[2], tempty[2], c0[8], drain, fix, c0r[4],
                          // inj, injdone, xch
  uint32_t tmem_slot;
  int32_t abort_flag;
  int32_t nbad_r, nbad_c, bad_row, bad_col;
  float fix_value;
  float inj_clean;
  float d_row, d_col;
  float tmax_a[4], tmax_b[4];  // per epilogue warp: partial tile maxima
  uint32_t epoch;              // this launch's flag value (workspace epoch + 1)
  int32_t epoch_ready;         // epoch published by the epilogue
};
static_assert(sizeof(Aux) <= kAuxBytes, "aux size");

__device__ __forceinline__ void record_error(const KernelParams& p, Aux* aux, int code) {
  atomicOr(&p.report->status_bits, 1u << code);
  atomicAdd(&p.report->timeouts, 1u);
  atomicExch(&aux->abort_flag, 1);
}

__device__ __forceinline__ bool aborted(Aux* aux) {
  return *(volatile int32_t*)&aux->abort_flag != 0;
}

// This launch's epoch as the epilogue publishes it in shared memory (the
// producer and MMA threads of an encode side CTA need its parity for the
// encode counter). Bounded: 0 after the limit, and the caller's counter
// wait then runs out and reports.
__device__ __forceinline__ uint32_t published_epoch(Aux* aux, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (*(volatile int32_t*)&aux->epoch_ready == 0)
    if (globaltimer() - t0 > limit_ns) return 0u;
  __threadfence_block();
  return *(volatile uint32_t*)&aux->epoch;
}

// Bounded mbarrier wait: true when the phase of `parity` completed; false
// on timeout or, if `honor_abort`, when another role of this CTA aborted.
// Drains (copies or MMAs this thread issued) pass honor_abort = false so
// they always wait for their own operations, up to the time limit.
static __device__ __noinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Aux* aux,
                                             uint64_t limit_ns, bool honor_abort = true,
                                             bool cluster_scope = false) {
  auto ready = [&]() {
    return cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (ready()) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ready()) return true;
    if ((i & 31) == 0) {
      if (honor_abort && aborted(aux)) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// wait_bar, inlined: loads issued before it stay in flight during the wait
// (a call would make the compiler wait for them first).
template <bool CLUSTER>
__device__ __forceinline__ bool try_wait_scoped(uint64_t* bar, uint32_t parity) {
  return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}

template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bar_inline(uint64_t* bar, uint32_t parity, Aux* aux,
                                                uint64_t limit_ns) {
  if (try_wait_scoped<CLUSTER>(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (try_wait_scoped<CLUSTER>(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (aborted(aux)) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ float f32_of(uint32_t u) { return __uint_as_float(u); }

// Fault injection (testing only). The flips of the slots that land in the
// 32-column chunk c32 of row r of 128 x BLK_N output tile `tile`, applied to
// v (slot 0 only when it is not applied inside the mainloop). Returns true
// when v changed; *clean gets the value before the first flip.
__device__ __forceinline__ bool apply_flips(const KernelParams& p, int tile, int r, int c32,
                                            float (&v)[32], float* clean) {
  bool hit = false;
#pragma unroll
  for (int sl = 0; sl < 2; ++sl) {
    if (p.inj_tile[sl] != tile || (sl == 0 && p.inj_kb >= 0)) continue;
    if (r != p.inj_row[sl] || (p.inj_col[sl] >> 5) != c32) continue;
    const int jc = p.inj_col[sl] & 31;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i == jc) {
        if (!hit && clean) *clean = v[i];
        v[i] = __uint_as_float(__float_as_uint(v[i]) ^ (1u << p.inj_bit[sl]));
      }
    hit = true;
  }
  return hit;
}

// Whether work item w runs slot 0's mid-mainloop MAC iteration (inj_kb) of
// the injected tile: for this CTA's 128-row half `half` of the item's tile,
// or (half < 0) for either half of a CTA pair's 256-row tile.
template <bool PAIR>
__device__ __forceinline__ bool mid_inject_item(const KernelParams& p, const Schedule& s,
                                                const Work& w, int half) {
  if (p.inj_kb < 0 || p.inj_tile[0] < 0 || w.tile < s.t_ck || p.inj_kb < w.kb_begin ||
      p.inj_kb >= w.kb_end)
    return false;
  int tm, tn;
  tile_coords(s, w.tile, tm, tn);
  const int tm0 = PAIR ? 2 * tm : tm;
  if (half >= 0) return p.inj_tile[0] == (tm0 + half) * s.tiles_n + tn;
  return p.inj_tile[0] == tm0 * s.tiles_n + tn ||
         (PAIR && p.inj_tile[0] == (tm0 + 1) * s.tiles_n + tn);
}

// First MAC iteration of a work item of n iterations under k staggering
// (offset from kb_begin; the item then wraps around to kb_begin).
__device__ __forceinline__ int stagger_offset(const KernelParams& p, int unit, int n) {
  return p.stagger > 1 ? (int)(((int64_t)(unit % p.stagger) * n) / p.stagger) : 0;
}

// The k order of one work item as at most three ascending ranges of MAC
// iterations, run one after the other: a staggered item runs
// [kb_begin + off, kb_end) then [kb_begin, kb_begin + off); a mid-mainloop
// injection at iteration inj_kb cuts the range that holds it after inj_kb
// (`pause` = the range after which the MMA thread waits for the flip). The
// loops over one range are the plain ascending k loops, so a launch without
// either option runs exactly one range per item with nothing extra per
// k-step.
struct KOrder {
  int lo0, hi0, lo1, hi1, lo2, hi2;
  int n, pause;
  __device__ __forceinline__ int lo(int r) const { return r == 0 ? lo0 : (r == 1 ? lo1 : lo2); }
  __device__ __forceinline__ int hi(int r) const { return r == 0 ? hi0 : (r == 1 ? hi1 : hi2); }
};

__device__ __forceinline__ KOrder k_order(int kb_begin, int kb_end, int off, int inj_kb) {
  KOrder o;
  o.lo0 = o.hi0 = o.lo1 = o.hi1 = o.lo2 = o.hi2 = 0;
  o.n = 0;
  o.pause = -1;
  auto push = [&](int a, int b) {
    if (o.n == 0) {
      o.lo0 = a;
      o.hi0 = b;
    } else if (o.n == 1) {
      o.lo1 = a;
      o.hi1 = b;
    } else {
      o.lo2 = a;
      o.hi2 = b;
    }
    ++o.n;
  };
  auto add = [&](int a, int b) {
    if (a >= b) return;
    if (inj_kb >= a && inj_kb < b) {
      push(a, inj_kb + 1);
      o.pause = o.n - 1;
      if (inj_kb + 1 < b) push(inj_kb + 1, b);
    } else {
      push(a, b);
    }
  };
  add(kb_begin + off, kb_end);
  add(kb_begin, kb_begin + off);
  return o;
}

// Sum over the 32 lanes of a warp for each of 32 columns: on return lane l
// holds the sum of column l (recursive halving, 31 shuffles).
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

template <int OUT>
__device__ __forceinline__ void pack_row(const float* y, uint32_t (&w)[32]);

template <>
__device__ __forceinline__ void pack_row<0>(const float* y, uint32_t (&w)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(y[i]);
}

template <>
__device__ __forceinline__ void pack_row<1>(const float* y, uint32_t (&w)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    __half2 h = __floats2half2_rn(y[2 * i], y[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

template <>
__device__ __forceinline__ void pack_row<2>(const float* y, uint32_t (&w)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int OUT>
__device__ __forceinline__ void unpack_row(const uint32_t (&w)[32], float* y);

template <>
__device__ __forceinline__ void unpack_row<0>(const uint32_t (&w)[32], float* y) {
#pragma unroll
  for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(w[i]);
}

template <>
__device__ __forceinline__ void unpack_row<1>(const uint32_t (&w)[32], float* y) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    float2 f = __half22float2(h);
    y[2 * i] = f.x;
    y[2 * i + 1] = f.y;
  }
}

template <>
__device__ __forceinline__ void unpack_row<2>(const uint32_t (&w)[32], float* y) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    float2 f = __bfloat1622float2(h);
    y[2 * i] = f.x;
    y[2 * i + 1] = f.y;
  }
}

// One 128-byte row of a staging buffer in the 128-byte swizzled order TMA
// uses: 16-byte chunk j of row r sits at chunk position j ^ (r % 8).
__device__ __forceinline__ void staging_write(uint8_t* buf, int r, const uint32_t (&w)[32]) {
  uint8_t* row = buf + r * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 q = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    *reinterpret_cast<uint4*>(row + ((j ^ (r & 7)) << 4)) = q;
  }
}

__device__ __forceinline__ void staging_read(const uint8_t* buf, int r, uint32_t (&w)[32]) {
  const uint8_t* row = buf + r * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 q = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
    w[4 * j] = q.x;
    w[4 * j + 1] = q.y;
    w[4 * j + 2] = q.z;
    w[4 * j + 3] = q.w;
  }
}

__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void st_cg_f4(float* p, float4 v) {
  __stcg(reinterpret_cast<float4*>(p), v);
}

// Partial tile layouts (per CTA slot). Output tiles (region 0) use one band
// per 32-row lane quadrant (32 x BN floats, contiguous, so an owner can pull
// a quadrant's partial with a single bulk copy); inside a band, 4-column
// groups of 32 rows: float index ((r / 32) * BN / 4 + c4) * 128 + (r % 32) * 4 + e.
// Checksum tiles (region 1) use only their first columns and keep them
// together: 4-column groups of all 128 rows, float index (c4 * 128 + r) * 4 + e.
// Either way the 32 lanes of a warp touch 512 contiguous bytes.
template <int BN>
__device__ __forceinline__ float* partial_at(float* slot, int c4, int r, bool band) {
  return band ? slot + ((size_t)((r >> 5) * (BN / 4) + c4) * 32 + (r & 31)) * 4
              : slot + ((size_t)c4 * kBM + r) * 4;
}
template <int BN>
constexpr uint32_t kPartialBandBytes = 32u * BN * 4u;

// LoadPartials for one 32-column chunk: v += the partials of peers
// first..last (ascending CTA order, so the sum is deterministic). Loads are
// issued four peers at a time before any is used, so an owner with many
// peers waits for one L2 round trip per group rather than per peer.
template <int BN>
__device__ __forceinline__ void add_peer_partials(float (&v)[32], float* partials, int first,
                                                  int last, int c32, int r, bool band,
                                                  int slot_stride = 1, int slot_offset = 0) {
  int peer = first;
  for (; peer + 3 <= last; peer += 4) {
    float4 t[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float* ps = partials + (size_t)((peer + u) * slot_stride + slot_offset) * kBM * BN;
#pragma unroll
      for (int j = 0; j < 8; ++j) t[u][j] = ld_cg_f4(partial_at<BN>(ps, c32 * 8 + j, r, band));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[4 * j] += t[u][j].x;
        v[4 * j + 1] += t[u][j].y;
        v[4 * j + 2] += t[u][j].z;
        v[4 * j + 3] += t[u][j].w;
      }
  }
  for (; peer <= last; ++peer) {
    float4 t[8];
    float* ps = partials + (size_t)(peer * slot_stride + slot_offset) * kBM * BN;
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = ld_cg_f4(partial_at<BN>(ps, c32 * 8 + j, r, band));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[4 * j] += t[j].x;
      v[4 * j + 1] += t[j].y;
      v[4 * j + 2] += t[j].z;
      v[4 * j + 3] += t[j].w;
    }
  }
}

// In-kernel encode pass: boxes of 64 rows x 256 k-columns (no swizzle). A
// unit is one operand tile (128 rows of A, enc_bn stored rows of B) x 256
// k-columns; side CTA sx of gs takes a contiguous range of units, split
// evenly in boxes.
constexpr int kEncInCols = 256;
constexpr int kEncInRows = 64;
constexpr int kEncInBoxBytes = kEncInCols * kEncInRows * 2;

__device__ __forceinline__ void enc_in_units(const KernelParams& p, int sx, int gs, int& u0,
                                             int& u1) {
  const int sub_a = kBM / kEncInRows, sub_b = p.enc_bn / kEncInRows;
  const int units_a = p.enc_tiles_a * p.enc_slices;
  const int units = units_a + p.enc_tiles_b * p.enc_slices;
  const int64_t boxes = (int64_t)units_a * sub_a + (int64_t)(units - units_a) * sub_b;
  auto first_unit_at = [&](int64_t box) -> int {
    const int64_t in_a = (int64_t)units_a * sub_a;
    if (box <= in_a) return (int)((box + sub_a - 1) / sub_a);
    return units_a + (int)((box - in_a + sub_b - 1) / sub_b);
  };
  u0 = first_unit_at(boxes * sx / gs);
  u1 = first_unit_at(boxes * (sx + 1) / gs);
}

__device__ __forceinline__ int enc_in_boxes(const KernelParams& p, int u0, int u1) {
  const int units_a = p.enc_tiles_a * p.enc_slices;
  int n = 0;
  for (int u = u0; u < u1; ++u) n += u < units_a ? kBM / kEncInRows : p.enc_bn / kEncInRows;
  return n;
}

// LoadPartials through the idle stage ring (one epilogue warp, its 32-row
// quadrant q of the tile): every peer's band of the quadrant in half-band
// pieces (two per peer), `slots` pieces in flight through
// `qring`, each folded into the accumulator columns in TMEM as it lands.
// bars[0, slots) are this warp's piece barriers (fresh: parities start at 0).
// Returns false after a timeout, with every copy it issued landed.
template <int BN>
static __device__ __noinline__ bool fixup_through_ring(uint8_t* qring, int slots,
                                                       const float* rpartials, int unit,
                                                       int peer_last, int slot_stride, int crank,
                                                       int q, int lane, uint32_t tacc,
                                                       uint64_t* bars, const KernelParams& p,
                                                       Aux* aux, uint64_t limit) {
  constexpr uint32_t kHalf = kPartialBandBytes<BN> / 2;
  const int items = 2 * (peer_last - unit);  // (peer, half) pieces
  auto issue = [&](int i) {
    const int sl = i % slots;
    const int slot_i = (unit + 1 + (i >> 1)) * slot_stride + crank;
    const float* src = rpartials + (size_t)slot_i * kBM * BN + (size_t)q * 32 * BN +
                       (size_t)(i & 1) * (kHalf / 4);
    mbar_arrive_expect_tx(&bars[sl], kHalf);
    bulk_load_g2s(qring + sl * kHalf, src, kHalf, &bars[sl]);
  };
  const int first = min(slots, items);
  if (lane == 0) {
    fence_proxy_async_global();
    for (int i = 0; i < first; ++i) issue(i);
  }
  __syncwarp();
  int issued = first;
  bool fine = true;
  int i = 0;
  for (; i < items; ++i) {
    const int sl = i % slots;
    fine = __all_sync(0xffffffffu, wait_bar(&bars[sl], (uint32_t)((i / slots) & 1), aux, limit));
    if (!fine) break;
    const int h = i & 1;
#pragma unroll 1
    for (int c32 = h * (BN / 64); c32 < (h + 1) * (BN / 64); ++c32) {
      uint32_t u[32];
      tmem_ld32(tacc + c32 * 32, u);
      const uint8_t* src = qring + sl * kHalf + (c32 - h * (BN / 64)) * 4096 + lane * 16;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float4 t = *reinterpret_cast<const float4*>(src + jj * 512);
        u[4 * jj] = __float_as_uint(f32_of(u[4 * jj]) + t.x);
        u[4 * jj + 1] = __float_as_uint(f32_of(u[4 * jj + 1]) + t.y);
        u[4 * jj + 2] = __float_as_uint(f32_of(u[4 * jj + 2]) + t.z);
        u[4 * jj + 3] = __float_as_uint(f32_of(u[4 * jj + 3]) + t.w);
      }
      tmem_st32(tacc + c32 * 32, u);
    }
    // The slot's reads are done (their values consumed) before lane 0 issues
    // its next copy.
    __syncwarp();
    if (lane == 0 && issued < items) issue(issued);
    issued += issued < items ? 1 : 0;
    __syncwarp();
  }
  if (!fine) {
    // Never leave with a copy in flight into the ring.
    if (lane == 0) {
      if (!aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
      for (int j = i; j < issued; ++j)
        wait_bar(&bars[j % slots], (uint32_t)((j / slots) & 1), aux, limit, false);
    }
    __syncwarp();
  }
  return fine;
}

// Split reduction, LoadPartials of one part: the partials of every other
// CTA covering the tile (owner .. contrib_last, ascending, without `unit`;
// the owner's in bank 2 when owner_bank2), restricted to this part's columns
// [col_lo, col_hi) of quadrant q's band, in pieces of at most BLK_N / 2
// columns through `slots` pipelined slots of `qring`, each folded into the
// accumulator columns in TMEM as it lands. bars[0, slots) are this warp's
// piece barriers (fresh). Returns false after a timeout, with every copy it
// issued landed.
template <int BN>
static __device__ __noinline__ bool fold_split_through_ring(
    uint8_t* qring, int slots, const float* rpartials, size_t bank2, int owner, int owner_bank2,
    int contrib_last, int unit, int slot_stride, int crank, int q, int lane, uint32_t tacc,
    int col_lo, int col_hi, uint64_t* bars, const KernelParams& p, Aux* aux, uint64_t limit) {
  constexpr int kPieceCols = BN / 2;
  constexpr uint32_t kSlotBytes = kPartialBandBytes<BN> / 2;
  const int npieces = (col_hi - col_lo + kPieceCols - 1) / kPieceCols;
  const int items = (contrib_last - owner) * npieces;  // other covers x pieces
  auto piece_cols = [&](int i, int& a, int& b) {
    a = col_lo + (i % npieces) * kPieceCols;
    b = min(col_hi, a + kPieceCols);
  };
  auto issue = [&](int i) {
    const int sl = i % slots;
    const int oi = i / npieces;
    const int u = owner + oi + (owner + oi >= unit ? 1 : 0);
    int a, b;
    piece_cols(i, a, b);
    const float* src = rpartials + (size_t)(u * slot_stride + crank) * kBM * BN +
                       (u == owner && owner_bank2 ? bank2 : 0) + (size_t)q * 32 * BN +
                       (size_t)a * 32;
    mbar_arrive_expect_tx(&bars[sl], (uint32_t)(b - a) * 128u);
    bulk_load_g2s(qring + sl * kSlotBytes, src, (uint32_t)(b - a) * 128u, &bars[sl]);
  };
  const int first = min(slots, items);
  if (lane == 0) {
    fence_proxy_async_global();
    for (int i = 0; i < first; ++i) issue(i);
  }
  __syncwarp();
  int issued = first;
  bool fine = true;
  int i = 0;
  for (; i < items; ++i) {
    const int sl = i % slots;
    fine = __all_sync(0xffffffffu, wait_bar(&bars[sl], (uint32_t)((i / slots) & 1), aux, limit));
    if (!fine) break;
    int a, b;
    piece_cols(i, a, b);
#pragma unroll 1
    for (int c32 = a / 32; c32 < b / 32; ++c32) {
      uint32_t u[32];
      tmem_ld32(tacc + c32 * 32, u);
      const uint8_t* src = qring + sl * kSlotBytes + (c32 * 32 - a) * 128 + lane * 16;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float4 t = *reinterpret_cast<const float4*>(src + jj * 512);
        u[4 * jj] = __float_as_uint(f32_of(u[4 * jj]) + t.x);
        u[4 * jj + 1] = __float_as_uint(f32_of(u[4 * jj + 1]) + t.y);
        u[4 * jj + 2] = __float_as_uint(f32_of(u[4 * jj + 2]) + t.z);
        u[4 * jj + 3] = __float_as_uint(f32_of(u[4 * jj + 3]) + t.w);
      }
      tmem_st32(tacc + c32 * 32, u);
    }
    __syncwarp();
    if (lane == 0 && issued < items) issue(issued);
    issued += issued < items ? 1 : 0;
    __syncwarp();
  }
  if (!fine) {
    if (lane == 0) {
      if (!aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
      for (int j = i; j < issued; ++j)
        wait_bar(&bars[j % slots], (uint32_t)((j / slots) & 1), aux, limit, false);
    }
    __syncwarp();
  }
  return fine;
}

// Elements of C in the launch's output type, one at a time or four at once
// (the shared tile reduction's plain loads and stores).
template <int OUT>
__device__ __forceinline__ float load_out(const void* c, int64_t i) {
  if constexpr (OUT == 0) return static_cast<const float*>(c)[i];
  else if constexpr (OUT == 1) return __half2float(static_cast<const __half*>(c)[i]);
  else return __bfloat162float(static_cast<const __nv_bfloat16*>(c)[i]);
}
template <int OUT>
__device__ __forceinline__ void store_out(void* c, int64_t i, float v) {
  if constexpr (OUT == 0) static_cast<float*>(c)[i] = v;
  else if constexpr (OUT == 1) static_cast<__half*>(c)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16*>(c)[i] = __float2bfloat16_rn(v);
}
template <int OUT>
__device__ __forceinline__ void unpack4(float4 w, float (&y)[4]) {
  y[0] = w.x;
  y[1] = w.y;
  y[2] = w.z;
  y[3] = w.w;
}
template <int OUT>
__device__ __forceinline__ void unpack4(uint2 w, float (&y)[4]) {
  const uint32_t h[2] = {w.x, w.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if constexpr (OUT == 1) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
      y[2 * i] = f.x;
      y[2 * i + 1] = f.y;
    } else {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&h[i]));
      y[2 * i] = f.x;
      y[2 * i + 1] = f.y;
    }
  }
}
template <int OUT, class Vec>
__device__ __forceinline__ Vec pack4(const float (&y)[4]) {
  if constexpr (OUT == 0) {
    return make_float4(y[0], y[1], y[2], y[3]);
  } else {
    uint32_t h[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if constexpr (OUT == 1) {
        const __half2 v = __floats2half2_rn(y[2 * i], y[2 * i + 1]);
        h[i] = *reinterpret_cast<const uint32_t*>(&v);
      } else {
        const __nv_bfloat162 v = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
        h[i] = *reinterpret_cast<const uint32_t*>(&v);
      }
    }
    return make_uint2(h[0], h[1]);
  }
}

// Shared LoadPartials + StoreTile (no ABFT): a tile covered by CTAs
// owner .. contrib_last of which owner .. part_last end their ranges in it.
// Each of those stored its whole partial and signalled (the owner in bank 2,
// the second region's flags and slots, when owner_bank2); after every
// cover's flag is set, participant j = unit - owner reduces its share of the tile's
// (32-row quadrant, 4-column group) items over all covers' partials in
// ascending CTA order, then applies alpha / beta and stores C with plain
// stores. The k=0 CTA no longer sums every peer alone, so no CTA of a deep,
// many-way split tile waits on one SM's read bandwidth. Called by all 128
// epilogue threads; false after a timeout.
template <class C>
static __device__ __noinline__ bool reduce_share(const KernelParams& p, float* rpartials,
                                                 uint32_t* rflags, int owner, int owner_bank2,
                                                 int contrib_last, int part_last, int unit,
                                                 int slot_stride, int crank, int m0, int n0,
                                                 int ew, int lane, uint32_t epoch, int out_tile,
                                                 Aux* aux, uint64_t limit) {
  constexpr int BN = C::BN;
  // Bank 2 of the owner's flag and partial slot.
  const size_t bank2 = (size_t)p.ws_ctas * kBM * BN;
  bool fine = true;
  if (ew == 0) {
    for (int u = owner + lane; u <= contrib_last && fine; u += 32) {
      if (u == unit) continue;
      const int fi = u * slot_stride + crank + (u == owner && owner_bank2 ? kMaxCtas : 0);
      if (ld_acquire_gpu(&rflags[fi]) == epoch) continue;
      const uint64_t t0 = globaltimer();
      uint32_t spins = 0;
      while (ld_acquire_gpu(&rflags[fi]) != epoch) {
        if (++spins > 64) nanosleep_ns(64);
        if ((spins & 15) == 0 && globaltimer() - t0 > limit) {
          record_error(p, aux, SKG_ERR_FIXUP_TIMEOUT);
          fine = false;
          break;
        }
      }
    }
  }
  if (!epi_all(fine && !aborted(aux))) return false;
  const int parts = part_last - owner + 1;
  const int j = unit - owner;
  const int items = 4 * (BN / 4);  // quadrant x 4-column group
  const int per = items / parts, extra = items % parts;
  const int ib = j * per + (j < extra ? j : extra);
  const int ie = ib + per + (j < extra ? 1 : 0);
  const int covers = contrib_last - owner + 1;
  // A warp takes items ib + ew, ib + ew + 4, ...; kBatch of them at a time
  // with their C0 values and kCov covers' partials in flight together, so
  // the loop waits for one round trip per batch and kCov covers. C0 and C
  // move as one 16-byte (fp32) or 8-byte (16-bit) vector per item and lane
  // when its four columns lie inside n.
  constexpr int kBatch = 2, kCov = 8;
  using Vec = typename std::conditional<C::OUT == 0, float4, uint2>::type;
  for (int t0 = ib + ew; t0 < ie; t0 += 4 * kBatch) {
    int64_t off[kBatch];
    int ncol[kBatch];  // columns of the item inside n (0 when the row is past m)
    float c0v[kBatch][4];
    float4 acc[kBatch];
#pragma unroll
    for (int bi = 0; bi < kBatch; ++bi) {
      const int t = t0 + 4 * bi;
      const int qi = t / (BN / 4), c4 = t - qi * (BN / 4);
      const int64_t gr = (int64_t)m0 + qi * 32 + lane;
      const int col = n0 + 4 * c4;
      acc[bi] = make_float4(0.f, 0.f, 0.f, 0.f);
      ncol[bi] = (t < ie && gr < p.m) ? max(0, min(4, p.n - col)) : 0;
      off[bi] = gr * p.ldc + col;
#pragma unroll
      for (int e = 0; e < 4; ++e) c0v[bi][e] = 0.f;
      if (p.beta != 0.f && ncol[bi] == 4) {
        const Vec w = *reinterpret_cast<const Vec*>(static_cast<const char*>(p.c_ptr) +
                                                    off[bi] * C::OUT_BYTES);
        unpack4<C::OUT>(w, c0v[bi]);
      } else if (p.beta != 0.f) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < ncol[bi]) c0v[bi][e] = load_out<C::OUT>(p.c_ptr, off[bi] + e);
      }
    }
    for (int cv0 = 0; cv0 < covers; cv0 += kCov) {
      float4 v[kBatch][kCov];
#pragma unroll
      for (int bi = 0; bi < kBatch; ++bi) {
        const int t = t0 + 4 * bi;
        const int qi = t / (BN / 4), c4 = t - qi * (BN / 4);
#pragma unroll
        for (int u = 0; u < kCov; ++u)
          if (t < ie && cv0 + u < covers)
            v[bi][u] = ld_cg_f4(partial_at<BN>(
                rpartials + (size_t)((owner + cv0 + u) * slot_stride + crank) * kBM * BN +
                    (cv0 + u == 0 && owner_bank2 ? bank2 : 0),
                c4, qi * 32 + lane, true));
      }
#pragma unroll
      for (int bi = 0; bi < kBatch; ++bi)
#pragma unroll
        for (int u = 0; u < kCov; ++u)
          if (t0 + 4 * bi < ie && cv0 + u < covers) {
            acc[bi].x += v[bi][u].x;
            acc[bi].y += v[bi][u].y;
            acc[bi].z += v[bi][u].z;
            acc[bi].w += v[bi][u].w;
          }
    }
#pragma unroll
    for (int bi = 0; bi < kBatch; ++bi) {
      if (ncol[bi] == 0) continue;
      const int t = t0 + 4 * bi;
      const int qi = t / (BN / 4), c4 = t - qi * (BN / 4);
      const int r = qi * 32 + lane;
      float y[4] = {acc[bi].x, acc[bi].y, acc[bi].z, acc[bi].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)  // fault injection (testing only)
          if (p.inj_tile[sl] == out_tile && !(sl == 0 && p.inj_kb >= 0) &&
              r == p.inj_row[sl] && 4 * c4 + e == p.inj_col[sl])
            y[e] = __uint_as_float(__float_as_uint(y[e]) ^ (1u << p.inj_bit[sl]));
        y[e] = p.alpha * y[e] + p.beta * c0v[bi][e];
      }
      if (ncol[bi] == 4) {
        *reinterpret_cast<Vec*>(static_cast<char*>(p.c_ptr) + off[bi] * C::OUT_BYTES) =
            pack4<C::OUT, Vec>(y);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < ncol[bi]) store_out<C::OUT>(p.c_ptr, off[bi] + e, y[e]);
      }
    }
  }
  return true;
}

// Eight consecutive 16-bit inputs (one 16-byte chunk of a stage row) as fp32.
template <bool F16>
__device__ __forceinline__ void unpack8_in(uint4 q, float (&x)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (F16) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    } else {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

// In-CTA ABFT references, for launches of at most one whole output tile per
// CTA ("Anatomy of High-Performance GEMM with Online Fault Tolerance on
// GPUs", threadblock-level FT-GEMM: the checksums are updated at every
// k-step from the operand tiles the block holds). For each stage of the
// tile the four epilogue warps read the A tile (128 rows) and the B tile (BN
// rows = output columns) out of shared memory (128-byte swizzle), form
//   e^T A_s (64 values: the stage's A rows summed) and B_s e (its B rows
//   summed), and accumulate in fp32
//   cr[r] += A_s[r, :] . (B_s e)    (row reference of the accumulator row r
//                                    the thread reads from TMEM),
//   cc[j] += (e^T A_s) . B_s[j, :]  (column references, j = r, r + 128),
// with the tile's max |a| and max |b| for the thresholds; every sum keeps
// eight independent chains. Then the stage goes back to the producer (its
// empty barrier counts the MMA commit and this arrival). `scratch` is 640
// floats of shared memory; the walk of the ring starts at (stage, phase)
// and the result says where it stands. ok = false after a timeout
// (recorded).
template <int BN>
struct LocalSums {
  float cr, cc[BN / 128], ma, mb;
  int stage;
  uint32_t phase;
  bool ok;
};

template <class C, bool F16>
static __device__ __noinline__ LocalSums<C::BN> local_checksums(
    const KernelParams& p, uint8_t* ring, uint64_t* full_bar, uint64_t* empty_bar, int stage,
    uint32_t phase, int nk, float* scratch, int ew, int lane, int et, int r, Aux* aux,
    uint64_t limit) {
  constexpr int BN = C::BN;
  const int ch = lane & 7;              // 16-byte chunk: k values 8 ch .. 8 ch + 7
  const int rg = ew * 4 + (lane >> 3);  // row group 0..15
  float* part = scratch;                // [warp][e^T A_s (64), B_s e (64)]
  float* fin = scratch + 4 * 128;       // e^T A_s (64), B_s e (64) of the whole CTA
  float cr8[8], cc8[BN / 128][8], ma8[8], mb8[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    cr8[e] = ma8[e] = mb8[e] = 0.f;
#pragma unroll
    for (int h = 0; h < BN / 128; ++h) cc8[h][e] = 0.f;
  }
  LocalSums<BN> out;
  out.ok = true;
  for (int kb = 0; kb < nk; ++kb) {
    const bool got = wait_bar(&full_bar[stage], phase, aux, limit);
    if (!got && !aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
    if (!epi_all(got && !aborted(aux))) {
      out.ok = false;
      break;
    }
    const uint8_t* sa = ring + stage * C::STAGE_BYTES;
    const uint8_t* sb = sa + C::A_BYTES;
    // Column sums of the stage: the thread's chunk over its row group.
    float as[8], bs[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) as[e] = bs[e] = 0.f;
#pragma unroll
    for (int i = 0; i < kBM / 16; ++i) {
      const int row = rg + 16 * i;
      float x[8];
      unpack8_in<F16>(
          *reinterpret_cast<const uint4*>(sa + row * 128 + ((ch ^ (row & 7)) << 4)), x);
#pragma unroll
      for (int e = 0; e < 8; ++e) as[e] += x[e];
    }
#pragma unroll
    for (int i = 0; i < BN / 16; ++i) {
      const int row = rg + 16 * i;
      float x[8];
      unpack8_in<F16>(
          *reinterpret_cast<const uint4*>(sb + row * 128 + ((ch ^ (row & 7)) << 4)), x);
#pragma unroll
      for (int e = 0; e < 8; ++e) bs[e] += x[e];
    }
    // The warp's four row groups (lane bits 3 and 4), then the four warps.
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      as[e] += __shfl_xor_sync(0xffffffffu, as[e], 8);
      bs[e] += __shfl_xor_sync(0xffffffffu, bs[e], 8);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      as[e] += __shfl_xor_sync(0xffffffffu, as[e], 16);
      bs[e] += __shfl_xor_sync(0xffffffffu, bs[e], 16);
    }
    if (lane < 8) {
      float4* pa = reinterpret_cast<float4*>(part + ew * 128 + ch * 8);
      float4* pb = reinterpret_cast<float4*>(part + ew * 128 + 64 + ch * 8);
      pa[0] = make_float4(as[0], as[1], as[2], as[3]);
      pa[1] = make_float4(as[4], as[5], as[6], as[7]);
      pb[0] = make_float4(bs[0], bs[1], bs[2], bs[3]);
      pb[1] = make_float4(bs[4], bs[5], bs[6], bs[7]);
    }
    named_bar_sync(1, kEpiThreads);
    fin[et] = (part[et] + part[128 + et]) + (part[256 + et] + part[384 + et]);
    named_bar_sync(1, kEpiThreads);
    // Row reference of row r against B_s e; column references of columns
    // r (+128) against e^T A_s.
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float x[8];
      unpack8_in<F16>(*reinterpret_cast<const uint4*>(sa + r * 128 + ((c ^ (r & 7)) << 4)), x);
      const float4 b0 = *reinterpret_cast<const float4*>(fin + 64 + 8 * c);
      const float4 b1 = *reinterpret_cast<const float4*>(fin + 64 + 8 * c + 4);
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cr8[e] = fmaf(x[e], bv[e], cr8[e]);
        ma8[e] = fmaxf(ma8[e], fabsf(x[e]));
      }
    }
#pragma unroll
    for (int h = 0; h < BN / 128; ++h) {
      const int j = r + 128 * h;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float x[8];
        unpack8_in<F16>(*reinterpret_cast<const uint4*>(sb + j * 128 + ((c ^ (j & 7)) << 4)),
                        x);
        const float4 a0 = *reinterpret_cast<const float4*>(fin + 8 * c);
        const float4 a1 = *reinterpret_cast<const float4*>(fin + 8 * c + 4);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          cc8[h][e] = fmaf(x[e], av[e], cc8[h][e]);
          mb8[e] = fmaxf(mb8[e], fabsf(x[e]));
        }
      }
    }
    named_bar_sync(1, kEpiThreads);  // every read of the stage and of fin is done
    if (et == 0) mbar_arrive(&empty_bar[stage]);
    if (++stage == C::STAGES) {
      stage = 0;
      phase ^= 1;
    }
  }
  out.cr = ((cr8[0] + cr8[1]) + (cr8[2] + cr8[3])) + ((cr8[4] + cr8[5]) + (cr8[6] + cr8[7]));
#pragma unroll
  for (int h = 0; h < BN / 128; ++h)
    out.cc[h] = ((cc8[h][0] + cc8[h][1]) + (cc8[h][2] + cc8[h][3])) +
                ((cc8[h][4] + cc8[h][5]) + (cc8[h][6] + cc8[h][7]));
  out.ma = fmaxf(fmaxf(fmaxf(ma8[0], ma8[1]), fmaxf(ma8[2], ma8[3])),
                 fmaxf(fmaxf(ma8[4], ma8[5]), fmaxf(ma8[6], ma8[7])));
  out.mb = fmaxf(fmaxf(fmaxf(mb8[0], mb8[1]), fmaxf(mb8[2], mb8[3])),
                 fmaxf(fmaxf(mb8[4], mb8[5]), fmaxf(mb8[6], mb8[7])));
  out.stage = stage;
  out.phase = phase;
  return out;
}

// Mid-mainloop fault injection (testing only), by the epilogue warp of lane
// quadrant q: wait until the MMAs up to the chosen iteration are done (inj),
// flip the bit in TMEM (accumulator columns at acc_base), record the value
// before and after in the report, and let the MMA thread go on (injdone, the
// leader's for a CTA pair).
template <bool PAIR>
static __device__ __noinline__ void mid_inject_flip(const KernelParams& p, uint32_t acc_base,
                                                    int q, int lane, uint64_t* inj_bar,
                                                    uint64_t* injdone_bar, Aux* aux,
                                                    uint64_t limit) {
  if (!__all_sync(0xffffffffu, wait_bar(inj_bar, 0, aux, limit, true, PAIR))) {
    if (lane == 0 && !aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
    return;
  }
  tc_fence_after();
  const uint32_t ta = acc_base + ((uint32_t)(q * 32) << 16) + (uint32_t)((p.inj_col[0] >> 5) * 32);
  uint32_t u[32];
  tmem_ld32(ta, u);
  if (lane == (p.inj_row[0] & 31)) {
    const int jc = p.inj_col[0] & 31;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i == jc) {
        const uint32_t before = u[i];
        u[i] ^= 1u << p.inj_bit[0];
        p.report->mid_before = __uint_as_float(before);
        p.report->mid_after = __uint_as_float(u[i]);
        atomicAdd(&p.report->mid_injected, 1u);
      }
  }
  tmem_st32(ta, u);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if constexpr (PAIR) mbar_arrive_cluster(cluster_addr(injdone_bar, 0));
    else mbar_arrive(injdone_bar);
  }
}

// Result of an output tile's ABFT check (check_tile): the located element
// and its corrected value (row < 0: none located).
struct TileFix {
  int row, col;
  float val;
};

// The ABFT check of one output tile in TMEM ("Anatomy of High-Performance
// GEMM with Online Fault Tolerance on GPUs", Fig. 3 (d)-(f)): thread r of the
// four epilogue warps sums accumulator row r (after adding the Stream-K
// peers' partials when add_partials, and, when `flips`, the testing flips,
// both written back to TMEM), the warps' column sums meet in their staging
// buffers, and each sum is compared with its reference (pf_*: the row
// checksum of row r, the column checksums of columns h * 128 + r, the
// encode pass's tile maxima and scales) under tau_row / tau_col. Exactly
// one mismatching row and column locate an element, whose value is
// recomputed from the row checksum and the rest of the row; any other
// mismatch is uncorrectable. Outcomes go to the report. The epilogue runs it
// before the tile's stores, or (a tile stored first) after them.
template <class C>
static __device__ __forceinline__ TileFix check_tile(
    const KernelParams& p, Aux* aux, uint8_t* epi, uint32_t tacc, int q, int lane, int et, int r,
    bool add_partials, float* rpartials, int unit, int peer_last, bool region0, int slot_stride,
    int crank, bool inject_here, bool flips, bool injected_tile, int out_tile, uint32_t epoch,
    float pf_ma, float pf_mb, float pf_cr0, float pf_cr1, const float* pf_cc0,
    const float* pf_cc1, int pf_ea, int pf_eb) {
  constexpr int BN = C::BN;
  auto colsum_of = [&](int qq) -> float* {
    const int ew_of_q = (qq + 2) & 3;  // warps 2..5 own quadrants 2, 3, 0, 1
    return reinterpret_cast<float*>(epi + ew_of_q * C::EPI_BUFS * C::EPI_BUF_BYTES);
  };
  TileFix fix{-1, -1, 0.f};
  // This warp's staging buffers hold its column sums below: its own
  // earlier TMA stores must have finished reading them.
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
  float* my_colsum = colsum_of(q);
  // The row sum in four interleaved partial sums: shorter dependency chains.
  float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int c32 = 0; c32 < BN / 32; ++c32) {
    uint32_t u[32];
    tmem_ld32(tacc + c32 * 32, u);
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = f32_of(u[i]);
    if (add_partials)
      add_peer_partials<BN>(v, rpartials, unit + 1, peer_last, c32, r, region0,
                            slot_stride, crank);
    // Fault injection (testing only): bits of fp32 accumulators,
    // after the fixup and before the check.
    bool inj_chunk = false;
    if (inject_here && flips) {
      float clean = 0.f;
      const bool hit = apply_flips(p, out_tile, r, c32, v, &clean);
      if (hit) aux->inj_clean = clean;
      inj_chunk = __any_sync(0xffffffffu, hit);
    }
    if (add_partials || inj_chunk) {
      uint32_t wv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) wv[i] = __float_as_uint(v[i]);
      tmem_st32(tacc + c32 * 32, wv);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) rs[i & 3] += v[i];
    my_colsum[c32 * 32 + lane] = warp_column_sums(v, lane);
  }
  const float rowsum = (rs[0] + rs[1]) + (rs[2] + rs[3]);
  // Reference checksums of this tile: thread r holds the row checksum
  // of row r and the column checksum of columns h*128 + r, each the
  // sum of its hi and lo partial products, unscaled by the tile's
  // power of two; tile maxima for the thresholds are the max over
  // the tile's encode units.
  const float cr = ldexpf(pf_cr0 + pf_cr1, -pf_eb);
  float cc[C::CC_GROUPS];
#pragma unroll
  for (int h = 0; h < C::CC_GROUPS; ++h) cc[h] = ldexpf(pf_cc0[h] + pf_cc1[h], -pf_ea);
  {
    float ma = pf_ma, mb = pf_mb;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, off));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    }
    if (lane == 0) {
      aux->tmax_a[q] = ma;
      aux->tmax_b[q] = mb;
    }
  }
  named_bar_sync(1, kEpiThreads);  // column sums and tile maxima stored
  // Default thresholds from the tile's own maxima:
  //   tau = 2^-12 sqrt(k) sqrt(side) max|A_tile| max|B_tile|.
  float tau_r = p.tau_row, tau_c = p.tau_col;
  {
    const float ma = fmaxf(fmaxf(aux->tmax_a[0], aux->tmax_a[1]),
                           fmaxf(aux->tmax_a[2], aux->tmax_a[3]));
    const float mb = fmaxf(fmaxf(aux->tmax_b[0], aux->tmax_b[1]),
                           fmaxf(aux->tmax_b[2], aux->tmax_b[3]));
    const float base = ldexpf(1.f, -12) * sqrtf((float)p.k) * ma * mb;
    if (!(tau_r > 0.f)) tau_r = base * sqrtf((float)BN);
    if (!(tau_c > 0.f)) tau_c = base * sqrtf((float)kBM);
  }
  if (et == 0) {  // the report keeps the largest thresholds used
    atomicMax(reinterpret_cast<int*>(&p.report->tau_row), __float_as_int(tau_r));
    atomicMax(reinterpret_cast<int*>(&p.report->tau_col), __float_as_int(tau_c));
  }

  const float d_r = rowsum - cr;
  const bool bad_r = !(fabsf(d_r) <= tau_r);
  float ratio_r = bad_r ? 0.f : fabsf(d_r) / tau_r;
  float ratio_c = 0.f;
  if (bad_r) {
    atomicAdd(&aux->nbad_r, 1);
    aux->bad_row = r;
    aux->d_row = d_r;
  }
#pragma unroll
  for (int h = 0; h < C::CC_GROUPS; ++h) {
    const int j = h * 128 + r;
    const float tot =
        colsum_of(0)[j] + colsum_of(1)[j] + colsum_of(2)[j] + colsum_of(3)[j];
    const float d_c = tot - cc[h];
    if (!(fabsf(d_c) <= tau_c)) {
      atomicAdd(&aux->nbad_c, 1);
      aux->bad_col = j;
      aux->d_col = d_c;
    } else {
      ratio_c = fmaxf(ratio_c, fabsf(d_c) / tau_c);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    ratio_r = fmaxf(ratio_r, __shfl_xor_sync(0xffffffffu, ratio_r, off));
    ratio_c = fmaxf(ratio_c, __shfl_xor_sync(0xffffffffu, ratio_c, off));
  }
  if (lane == 0) {
    atomicMax(reinterpret_cast<int*>(&p.report->max_ratio_row), __float_as_int(ratio_r));
    atomicMax(reinterpret_cast<int*>(&p.report->max_ratio_col), __float_as_int(ratio_c));
  }
  named_bar_sync(1, kEpiThreads);  // mismatch counts complete

  const int nbr = aux->nbad_r, nbc = aux->nbad_c;
  const int brow = aux->bad_row, bcol = aux->bad_col;
  const bool single = (nbr == 1 && nbc == 1);
  if (et == 0) atomicAdd(&p.report->tiles_checked, 1u);
  if (single && (brow >> 5) == q) {
    // Locate at (brow, bcol); recompute the value from the row
    // checksum and the rest of the row (survives Inf / NaN).
    float rest = 0.f, before = 0.f;
#pragma unroll 1
    for (int c32 = 0; c32 < BN / 32; ++c32) {
      uint32_t u[32];
      tmem_ld32(tacc + c32 * 32, u);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x = f32_of(u[i]);
        if (c32 * 32 + i == bcol) before = x;
        else rest += x;
      }
    }
    if (r == brow) {
      const float after = cr - rest;
      aux->fix_value = after;
      atomicAdd(&p.report->detected, 1u);
      atomicAdd(&p.report->corrected, 1u);
      atomicOr(&p.report->status_bits, 1u << SKG_ABFT_CORRECTED);
      const uint32_t idx = atomicAdd(&p.report->n_records, 1u);
      if (idx < SKG_MAX_RECORDS) {
        skg_fault_record_t* rec = &p.report->records[idx];
        rec->launch = epoch;
        rec->tile = out_tile;
        rec->row = brow;
        rec->col = bcol;
        rec->status = SKG_ABFT_CORRECTED;
        rec->n_bad_rows = nbr;
        rec->n_bad_cols = nbc;
        rec->injected = injected_tile ? 1u : 0u;
        rec->before = before;
        rec->after = after;
        rec->delta_row = aux->d_row;
        rec->delta_col = aux->d_col;
        rec->clean_value = inject_here ? aux->inj_clean : 0.f;
      }
    }
  } else if (!single && (nbr != 0 || nbc != 0) && et == 0) {
    atomicAdd(&p.report->detected, 1u);
    atomicAdd(&p.report->uncorrectable, 1u);
    atomicOr(&p.report->status_bits, 1u << SKG_ABFT_UNCORRECTABLE);
    const uint32_t idx = atomicAdd(&p.report->n_records, 1u);
    if (idx < SKG_MAX_RECORDS) {
      skg_fault_record_t* rec = &p.report->records[idx];
      rec->launch = epoch;
      rec->tile = out_tile;
      rec->row = nbr == 1 ? brow : -1;
      rec->col = nbc == 1 ? bcol : -1;
      rec->status = SKG_ABFT_UNCORRECTABLE;
      rec->n_bad_rows = nbr;
      rec->n_bad_cols = nbc;
      rec->injected = injected_tile ? 1u : 0u;
      rec->before = 0.f;
      rec->after = 0.f;
      rec->delta_row = nbr ? aux->d_row : 0.f;
      rec->delta_col = nbc ? aux->d_col : 0.f;
      rec->clean_value = inject_here ? aux->inj_clean : 0.f;
    }
  }
  named_bar_sync(1, kEpiThreads);  // corrected value published
  if (single) {
    fix.row = brow;
    fix.col = bcol;
    fix.val = aux->fix_value;
  }
  named_bar_sync(1, kEpiThreads);  // everyone has read the decision
  if (et == 0) {
    aux->nbad_r = 0;
    aux->nbad_c = 0;
    aux->bad_row = -1;
    aux->bad_col = -1;
  }
  return fix;
}

template <class C>
__global__ void __launch_bounds__(kThreads, 1)
    skg_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmB128,
                    const __grid_constant__ CUtensorMap tmBE,
                    const __grid_constant__ CUtensorMap tmEA,
                    const __grid_constant__ CUtensorMap tmCr,
                    const __grid_constant__ CUtensorMap tmCc,
                    const __grid_constant__ CUtensorMap tmEncA,
                    const __grid_constant__ CUtensorMap tmEncB, const KernelParams p) {
  constexpr int BN = C::BN;
  constexpr int STAGES = C::STAGES;
  constexpr int ACC_BUFS = C::ACC_BUFS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* epi = ring + STAGES * C::STAGE_BYTES;
  Aux* aux = reinterpret_cast<Aux*>(epi + C::EPI_BYTES);
  uint64_t* full_bar = aux->bars;
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* c0_bar = tempty_bar + 2;  // [epilogue warp][staging buffer]: C0 rows landed
  uint64_t* drain_bar = c0_bar + 8;
  uint64_t* fix_bar = drain_bar + 1;  // [epilogue warp][slot]: staged peer partials
  uint64_t* c0r_bar = fix_bar + 4 * kFixSlots;  // per epilogue warp: C0 staged in the ring
  // Mid-mainloop fault injection: the MMAs up to the chosen iteration are
  // done (inj), the flipped value is back in TMEM (injdone, the leader's).
  uint64_t* inj_bar = c0r_bar + 4;
  uint64_t* injdone_bar = inj_bar + 1;
  // ILC with CTA pairs: the peer's column checksums have landed in xbuf.
  uint64_t* xch_bar = injdone_bar + 1;
  static_assert(2 * 8 + 2 + 2 + 8 + 1 + 4 * kFixSlots + 4 + 2 + 1 <= 60, "barrier slots");
  float* xbuf = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(aux) + C::AUX_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Schedule& s = p.s;
  const uint64_t limit = p.timeout_ns;
  // CTA pairs: rank within the cluster (0 = leader, which issues the MMAs)
  // and the schedule's CTA index, shared by both CTAs of a pair.
  const uint32_t crank = C::PAIR ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const int unit = C::PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  // This CTA's flag and partial slot, and its row offset inside a tile.
  const int slot_stride = C::PAIR ? 2 : 1;
  const int my_slot_idx = unit * slot_stride + (int)crank;
  const int row_half = (int)crank * kBM;
  constexpr int kCkHalf = C::PAIR ? 2 : 1;  // 128-row checksum tiles per side tile
  // Dedicated side CTA that first runs its share of the encode pass.
  const bool enc_here = C::ABFT && !C::PAIR && p.enc_inkernel && (int)blockIdx.x >= s.g;
  static_assert(!C::ABFT || C::STAGE_BYTES >= kEncInBoxBytes, "an encode box fills one ring stage");

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmC);
      if (C::ABFT && p.s.t_ck > 0) {
        prefetch_tmap(&tmB128);
        prefetch_tmap(&tmBE);
        prefetch_tmap(&tmEA);
        prefetch_tmap(&tmCr);
        prefetch_tmap(&tmCc);
      }
      aux->abort_flag = 0;
      aux->nbad_r = aux->nbad_c = 0;
      aux->bad_row = aux->bad_col = -1;
      aux->epoch_ready = 0;
    }
    // The barriers in one go, a lane each: every one counts a single
    // arrival except the accumulator-empty ones, which the epilogue threads
    // release (both CTAs' for a pair).
    const int nbars = (int)(xch_bar + 1 - full_bar);
    for (int i = lane; i < nbars; i += 32) {
      uint64_t* bar = full_bar + i;
      const bool acc_empty = bar >= tempty_bar && bar < tempty_bar + 2;
      // The exchange barrier counts the peer's 128 epilogue threads.
      if (bar == xch_bar) {
        mbar_init(bar, kEpiThreads);
        continue;
      }
      // In-CTA ABFT: the epilogue also reads every stage, so a stage is
      // free once the MMA commit and the epilogue have both arrived.
      const bool stage_empty = bar >= empty_bar && bar < empty_bar + STAGES;
      mbar_init(bar, acc_empty ? (C::PAIR ? 2 * kEpiThreads : kEpiThreads)
                               : ((C::LOCAL && stage_empty) ? 2 : 1));
    }
    fence_barrier_init();
  }
  if constexpr (C::ILC) {
    // Encoding slots: the TMA writes rows 0 and 1 of each (hi, lo); the
    // other rows stay zero for the N = 16 checksum MMAs that read them.
    constexpr int kSlotChunks = 2 * C::ENC_SLOT_BYTES / 16;
    for (int i = threadIdx.x; i < STAGES * kSlotChunks; i += kThreads)
      *reinterpret_cast<uint4*>(ring + (i / kSlotChunks) * C::STAGE_BYTES + C::ENCA_OFF +
                                (i % kSlotChunks) * 16) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    if constexpr (C::PAIR) {
      tmem_alloc_pair(&aux->tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&aux->tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  // A pair's barriers must be initialised before the peer signals them.
  if constexpr (C::PAIR) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = aux->tmem_slot;
  uint32_t ticket = 0;  // this CTA's launch ticket (taken by epilogue thread 0)
  // Everything above touched only this CTA's shared memory and TMEM; from
  // here on the kernel reads the previous kernel's outputs (inputs, ABFT
  // checksums, the workspace epoch).
  griddep_wait();
  if (threadIdx.x == 0) {
    griddep_launch_dependents();
    if (p.cta_clock) p.cta_clock[2 * blockIdx.x] = globaltimer();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Cursor cur;
      cur.init(s, unit);
      Work w;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pending = 0;  // bit i: stage i has a load this thread issued
      uint32_t pend_par = 0; // parity of that load's phase
      bool ok = true;
      if (enc_here) {
        // Encode pass: this side CTA's units, one box per ring stage.
        if (threadIdx.x == 0) {
          prefetch_tmap(&tmEncA);
          prefetch_tmap(&tmEncB);
        }
        int u0, u1;
        enc_in_units(p, (int)blockIdx.x - s.g, s.g_ck, u0, u1);
        const int units_a = p.enc_tiles_a * p.enc_slices;
        for (int u = u0; ok && u < u1; ++u) {
          const bool is_a = u < units_a;
          const int t = u / p.enc_slices, sl = u - t * p.enc_slices;
          const CUtensorMap* map = is_a ? &tmEncA : &tmEncB;
          const int row0 = is_a ? t * kBM : (t - p.enc_tiles_a) * p.enc_bn;
          const int nsub = is_a ? kBM / kEncInRows : p.enc_bn / kEncInRows;
          for (int h = 0; h < nsub; ++h) {
            if (!mbar_try_wait(&empty_bar[stage], phase ^ 1) &&
                !wait_bar(&empty_bar[stage], phase ^ 1, aux, limit)) {
              if (!aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full_bar[stage], kEncInBoxBytes);
            tma_load_2d(ring + stage * C::STAGE_BYTES, map, &full_bar[stage], sl * kEncInCols,
                        row0 + h * kEncInRows);
            pending |= 1u << stage;
            pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        // The checksum tiles read every side CTA's encodings: wait for all.
        if (ok) {
          const uint32_t par = (published_epoch(aux, limit) - 1u) & 1u;
          const uint64_t t0 = globaltimer();
          while (ld_acquire_gpu(&p.hdr->enc_done[par]) < (uint32_t)s.g_ck) {
            nanosleep_ns(64);
            if (globaltimer() - t0 > limit) {
              if (!aborted(aux)) record_error(p, aux, SKG_ERR_FIXUP_TIMEOUT);
              ok = false;
              break;
            }
          }
          // Written through the generic proxy, read by TMA (async proxy).
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
      }
      while (ok && cur.next(s, w)) {
        // Operand maps and row coordinates of this tile: an output tile, or
        // a tile of one of the fused checksum GEMMs.
        const CUtensorMap* mapA = &tmA;
        const CUtensorMap* mapB = &tmB;
        uint32_t tx = C::TX_BYTES;
        int kpack = 1;
        int rowA, rowB;
        int enc_ra = 0, enc_rb = 0;  // ILC: hi rows of this CTA's e^T A and the tile's B e
        bool amn = C::MN && p.a_mn != 0, bmn = C::MN && p.b_mn != 0;  // MN-major boxes
        if (w.tile >= s.t_ck) {
          int tm, tn;
          tile_coords(s, w.tile, tm, tn);
          rowA = tm * (C::PAIR ? 2 * kBM : kBM) + row_half;
          rowB = tn * BN + (C::PAIR ? (int)crank * C::B_ROWS : 0);
          enc_ra = kEncRows * (rowA / kBM);
          enc_rb = kEncRows * tn;
        } else if (w.tile < p.ck_cr_tiles) {
          bmn = false;
          // Checksum tile: the encoding box holds only the rows the MMA uses.
          mapB = &tmBE;
          rowA = (w.tile * kCkHalf + (int)crank) * kBM;
          rowB = (int)crank * (p.ck_rows_cr / kCkHalf);
          tx = C::A_BYTES + p.ck_rows_cr / kCkHalf * kBK * 2;
          kpack = C::CK_PACK ? p.ck_kpack_cr : 1;
        } else {
          amn = p.b_mn != 0;
          bmn = false;
          mapA = &tmB128;
          mapB = &tmEA;
          rowA = ((w.tile - p.ck_cr_tiles) * kCkHalf + (int)crank) * kBM;
          rowB = (int)crank * (p.ck_rows_cc / kCkHalf);
          tx = C::A_BYTES + p.ck_rows_cc / kCkHalf * kBK * 2;
          kpack = C::CK_PACK ? p.ck_kpack_cc : 1;
        }
        // The k-loop, compiled once per operand-layout pair so that no
        // layout branch sits in the loop (a runtime one cost 5-9 %); the
        // K-major instantiations compile only the K-major copy (more copies
        // in one kernel cost ~1.3 us at 2048^3 through code size).
        auto k_loop = [&](auto a_tag, auto b_tag) {
          constexpr bool a_box = decltype(a_tag)::value, b_box = decltype(b_tag)::value;
          // k order: the item's ranges (the MMA thread walks the same ones).
          const KOrder ko =
              k_order(w.kb_begin, w.kb_end,
                      w.tile >= s.t_ck ? stagger_offset(p, unit, w.kb_end - w.kb_begin) : 0, -1);
          for (int rg = 0; rg < ko.n && ok; ++rg)
          for (int kb = ko.lo(rg), kb_hi = ko.hi(rg); kb < kb_hi; kb += kpack) {
            if (!try_wait_scoped<C::PAIR>(&empty_bar[stage], phase ^ 1) &&
                !wait_bar(&empty_bar[stage], phase ^ 1, aux, limit, true, C::PAIR)) {
              if (!aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
              ok = false;
              break;
            }
            uint8_t* st = ring + stage * C::STAGE_BYTES;
            if constexpr (C::PAIR) {
              // Both CTAs' copies complete on the leader's full barrier; the
              // leader expects the pair's bytes.
              const uint32_t fb = cluster_addr(&full_bar[stage], 0);
              // ILC: both CTAs load their e^T A rows, the leader the tile's B e.
              if (leader)
                mbar_arrive_expect_tx(&full_bar[stage], 2 * tx + (C::ILC ? 3 * C::ENC_BOX_BYTES : 0));
              if constexpr (C::ILC) {
                tma_load_2d_pair(st + C::ENCA_OFF, &tmEA, fb, kb * kBK, enc_ra);
                if (leader) tma_load_2d_pair(st + C::ENCB_OFF, &tmBE, fb, kb * kBK, enc_rb);
              }
              if constexpr (!a_box) {
                tma_load_2d_pair(st, mapA, fb, kb * kBK, rowA);
              } else {
                for (int h = 0; h < kBM / kMnBox; ++h)
                  tma_load_2d_pair(st + h * kMnBoxBytes, mapA, fb, rowA + h * kMnBox, kb * kBK);
              }
              if constexpr (!b_box) {
                tma_load_2d_pair(st + C::A_BYTES, mapB, fb, kb * kBK, rowB);
              } else {
                for (int h = 0; h < C::B_ROWS / kMnBox; ++h)
                  tma_load_2d_pair(st + C::A_BYTES + h * kMnBoxBytes, mapB, fb, rowB + h * kMnBox,
                                   kb * kBK);
              }
            } else if (kpack == 1) {
              mbar_arrive_expect_tx(&full_bar[stage], tx + (C::ILC ? 2 * C::ENC_BOX_BYTES : 0));
              if constexpr (C::ILC) {
                tma_load_2d(st + C::ENCA_OFF, &tmEA, &full_bar[stage], kb * kBK, enc_ra);
                tma_load_2d(st + C::ENCB_OFF, &tmBE, &full_bar[stage], kb * kBK, enc_rb);
              }
              if constexpr (!a_box) {
                tma_load_2d(st, mapA, &full_bar[stage], kb * kBK, rowA);
              } else {
                for (int h = 0; h < kBM / kMnBox; ++h)
                  tma_load_2d(st + h * kMnBoxBytes, mapA, &full_bar[stage], rowA + h * kMnBox,
                              kb * kBK);
              }
              if constexpr (!b_box) {
                tma_load_2d(st + C::A_BYTES, mapB, &full_bar[stage], kb * kBK, rowB);
              } else {
                for (int h = 0; h < C::B_ROWS / kMnBox; ++h)
                  tma_load_2d(st + C::A_BYTES + h * kMnBoxBytes, mapB, &full_bar[stage],
                              rowB + h * kMnBox, kb * kBK);
              }
            } else {  // packed checksum stage
              const int nk = min(2, w.kb_end - kb);
              mbar_arrive_expect_tx(&full_bar[stage], tx * nk);
              for (int j = 0; j < nk; ++j) {
                if constexpr (!a_box) {
                  tma_load_2d(st + j * C::A_BYTES, mapA, &full_bar[stage], (kb + j) * kBK, rowA);
                } else {
                  for (int h = 0; h < kBM / kMnBox; ++h)
                    tma_load_2d(st + j * C::A_BYTES + h * kMnBoxBytes, mapA, &full_bar[stage],
                                rowA + h * kMnBox, (kb + j) * kBK);
                }
                tma_load_2d(st + 2 * C::A_BYTES + j * C::ENC_SLOT, mapB, &full_bar[stage],
                            (kb + j) * kBK, rowB);
              }
            }
            if (leader) {
              pending |= 1u << stage;
              pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        };
        if constexpr (!C::MN) {
          k_loop(std::false_type{}, std::false_type{});
        } else if (amn) {
          if (bmn) k_loop(std::true_type{}, std::true_type{});
          else k_loop(std::true_type{}, std::false_type{});
        } else {
          if (bmn) k_loop(std::false_type{}, std::true_type{});
          else k_loop(std::false_type{}, std::false_type{});
        }
      }
      // Never leave with a copy in flight into this CTA's shared memory.
      for (int i = 0; i < STAGES; ++i)
        if (pending & (1u << i)) wait_bar(&full_bar[i], (pend_par >> i) & 1, aux, limit, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (one thread; in a CTA pair only the leader's issues, for both CTAs)
    if (lane == 0 && leader) {
      // Shared-memory descriptor of the ring's first byte; the ring lies in
      // the first 256 KB of shared memory, so adding (offset >> 4) to the
      // 14-bit address field never carries out of it.
      const uint64_t ring_desc = sdesc_sw128(smem_u32(ring));
      // MN-major operands: leading byte offset = the distance between the
      // 64-element MN boxes (the K-major descriptor carries 1 there), and a
      // 16-k slice is two 8-row groups of 1024 bytes.
      const uint64_t mn_lbo = (uint64_t)((kMnBoxBytes >> 4) - 1) << 16;
      Cursor cur;
      cur.init(s, unit);
      Work w;
      int stage = 0;
      uint32_t phase = 0;
      int ab = 0;
      uint32_t aphase = 0;
      bool ok = true;
      bool issued = false;
      if (enc_here) {
        // The ring's first stages carry this CTA's encode boxes. Start only
        // once every side CTA's encode pass is done: by then all of this
        // CTA's boxes have landed and been consumed, so the first wait below
        // cannot mistake an earlier phase of a stage for the one it wants
        // (a parity wait only tells phases apart one at a time).
        int u0, u1;
        enc_in_units(p, (int)blockIdx.x - s.g, s.g_ck, u0, u1);
        const int nb = enc_in_boxes(p, u0, u1);
        stage = nb % STAGES;
        phase = (uint32_t)((nb / STAGES) & 1);
        const uint32_t par = (published_epoch(aux, limit) - 1u) & 1u;
        const uint64_t t0 = globaltimer();
        while (ld_acquire_gpu(&p.hdr->enc_done[par]) < (uint32_t)s.g_ck) {
          nanosleep_ns(64);
          if (globaltimer() - t0 > limit) {
            if (!aborted(aux)) record_error(p, aux, SKG_ERR_FIXUP_TIMEOUT);
            ok = false;
            break;
          }
        }
      }
      while (ok && cur.next(s, w)) {
        if (!wait_bar(&tempty_bar[ab], aphase ^ 1, aux, limit, true, C::PAIR)) {
          if (!aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + ab * C::ACC_COLS;
        const uint32_t idesc = w.tile >= s.t_ck ? p.idesc_main
                               : (w.tile < p.ck_cr_tiles ? p.idesc_cr : p.idesc_cc);
        const int kpack = (!C::CK_PACK || w.tile >= s.t_ck)
                              ? 1
                              : (w.tile < p.ck_cr_tiles ? p.ck_kpack_cr : p.ck_kpack_cc);
        // MN-major operands of this item (the producer's choice, above).
        const bool amn = C::MN && (w.tile >= s.t_ck ? p.a_mn != 0
                                                    : (w.tile < p.ck_cr_tiles ? p.a_mn != 0
                                                                              : p.b_mn != 0));
        const bool bmn = C::MN && w.tile >= s.t_ck && p.b_mn != 0;
        const uint64_t a_lbo = amn ? mn_lbo : 0, b_lbo = bmn ? mn_lbo : 0;
        const int a_step = amn ? (2048 >> 4) : 2, b_step = bmn ? (2048 >> 4) : 2;
        if (kpack == 1) {
          // One k-step of MMAs (and, ILC, its checksum MMAs); false after a
          // timeout. kb_first is the item's first k-step, whose first MMA
          // starts the accumulator.
          auto mma_kstep = [&](int kb, int kb_first) -> bool {
            // Inline fast path: the stage is usually full already.
            if (!mbar_try_wait(&full_bar[stage], phase) &&
                !wait_bar(&full_bar[stage], phase, aux, limit)) {
              if (!aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
              ok = false;
              return false;
            }
            tc_fence_after();
            // Descriptors advance linearly with the (16-byte granular)
            // address: by 32 bytes per 16-k slice inside a K-major 128-byte
            // row, or by two 8-row k groups (2048 bytes) of an MN-major box.
            const uint64_t ad0 = ring_desc + (uint64_t)((stage * C::STAGE_BYTES) >> 4) + a_lbo;
            const uint64_t bd0 = ring_desc +
                                 (uint64_t)((stage * C::STAGE_BYTES + C::A_BYTES) >> 4) + b_lbo;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint32_t acc = (kb != kb_first || kk > 0) ? 1u : 0u;
              const uint64_t ad = ad0 + (uint64_t)(kk * a_step), bd = bd0 + (uint64_t)(kk * b_step);
              if constexpr (C::PAIR) umma_f16_pair(d, ad, bd, idesc, acc);
              else umma_f16(d, ad, bd, idesc, acc);
            }
            if constexpr (C::ILC) {
              // The reference checksums of this k-step: cr += A_s (B e)_s
              // (A as the A operand, the B e rows as N) and cc += B_s
              // (e^T A)_s (B's rows as the A operand, the e^T A rows as N).
              const uint64_t ea0 = ring_desc + (uint64_t)((stage * C::STAGE_BYTES + C::ENCA_OFF) >> 4);
              const uint64_t eb0 = ring_desc + (uint64_t)((stage * C::STAGE_BYTES + C::ENCB_OFF) >> 4);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint32_t acc = (kb != kb_first || kk > 0) ? 1u : 0u;
                if constexpr (C::PAIR) {
                  umma_f16_pair(d + C::CR_COL, ad0 + kk * 2, eb0 + kk * 2, p.idesc_cr, acc);
                  umma_f16_pair(d + C::CC_COL, bd0 + kk * 2, ea0 + kk * 2, p.idesc_cc, acc);
                } else {
                  umma_f16(d + C::CR_COL, ad0 + kk * 2, eb0 + kk * 2, p.idesc_cr, acc);
                  umma_f16(d + C::CC_COL, bd0 + kk * 2, ea0 + kk * 2, p.idesc_cc, acc);
                }
              }
            }
            issued = true;
            if constexpr (C::PAIR) umma_commit_pair(&empty_bar[stage]);  // both CTAs' stage
            else umma_commit(&empty_bar[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
            return true;
          };
          const int koff =
              w.tile >= s.t_ck ? stagger_offset(p, unit, w.kb_end - w.kb_begin) : 0;
          const int inj_kb_here = mid_inject_item<C::PAIR>(p, s, w, -1) ? p.inj_kb : -1;
          if (koff == 0 && inj_kb_here < 0) {
            // The plain ascending k loop: every launch without k staggering
            // or a mid-mainloop flip.
            for (int kb = w.kb_begin; kb < w.kb_end; ++kb)
              if (!mma_kstep(kb, w.kb_begin)) break;
          } else {
            // The producer's k ranges (staggered start, wrap-around), cut
            // after a mid-mainloop injection's iteration.
            const KOrder ko = k_order(w.kb_begin, w.kb_end, koff, inj_kb_here);
            for (int rg = 0; rg < ko.n && ok; ++rg) {
              for (int kb = ko.lo(rg), kb_hi = ko.hi(rg); kb < kb_hi; ++kb)
                if (!mma_kstep(kb, ko.lo0)) break;
              if (ok && rg == ko.pause) {
                // Mid-mainloop fault injection (testing only): once these MMAs
                // are done, the epilogue warp of the row's lane quadrant flips
                // the value in TMEM; the next MMAs accumulate onto it.
                if constexpr (C::PAIR) umma_commit_pair(inj_bar);
                else umma_commit(inj_bar);
                if (!wait_bar(injdone_bar, 0, aux, limit, true, C::PAIR)) {
                  if (!aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
                  ok = false;
                }
                tc_fence_after();
              }
            }
          }
        } else {
          // Packed checksum stages: A(k), A(k+1), enc(k), enc(k+1).
          for (int kb = w.kb_begin; kb < w.kb_end; kb += 2) {
            if (!wait_bar(&full_bar[stage], phase, aux, limit)) {
              if (!aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st_addr = smem_u32(ring + stage * C::STAGE_BYTES);
            const int nk = min(2, w.kb_end - kb);
            for (int j = 0; j < nk; ++j) {
              const uint32_t a_addr = st_addr + j * C::A_BYTES;
              const uint32_t b_addr = st_addr + 2 * C::A_BYTES + j * C::ENC_SLOT;
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk) {
                const uint64_t ad = sdesc_sw128(a_addr) + a_lbo + (uint64_t)(kk * a_step);
                const uint64_t bd = sdesc_sw128(b_addr + kk * 32);
                const uint32_t acc = (kb > w.kb_begin || j > 0 || kk > 0) ? 1u : 0u;
                umma_f16(d, ad, bd, idesc, acc);
              }
            }
            issued = true;
            umma_commit(&empty_bar[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        if (!ok) break;
        if constexpr (C::PAIR) umma_commit_pair(&tfull_bar[ab]);  // both CTAs' accumulator
        else umma_commit(&tfull_bar[ab]);
        if (++ab == ACC_BUFS) {
          ab = 0;
          aphase ^= 1;
        }
      }
      if (issued) {
        // All MMAs this thread issued complete before TMEM is released.
        if constexpr (C::PAIR) umma_commit_pair(drain_bar);
        else umma_commit(drain_bar);
        wait_bar(drain_bar, 0, aux, limit, false, C::PAIR);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;         // epilogue warp 0..3
    const int q = warp & 3;          // TMEM lane quadrant
    const int r = q * 32 + lane;     // tile row of this thread
    const int et = threadIdx.x - 64; // epilogue thread 0..127
    uint8_t* ebuf = epi + ew * C::EPI_BUFS * C::EPI_BUF_BYTES;
    // Column partial sums of the warp owning lane quadrant qq.
    auto colsum_of = [&](int qq) -> float* {
      const int ew_of_q = (qq + 2) & 3;  // warps 2..5 own quadrants 2, 3, 0, 1
      return reinterpret_cast<float*>(epi + ew_of_q * C::EPI_BUFS * C::EPI_BUF_BYTES);
    };
    // This launch's epoch: read once, published to the other roles, then
    // this CTA's ticket (its value is first used at the CTA's exit, so the
    // round trip stays off every path).
    if (et == 0) {
      aux->epoch = ld_acquire_gpu(&p.hdr->epoch) + 1u;
      __threadfence_block();
      *reinterpret_cast<volatile int32_t*>(&aux->epoch_ready) = 1;
    }
    named_bar_sync(1, kEpiThreads);
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t*>(&aux->epoch);
    const uint32_t par = (epoch - 1u) & 1u;  // this launch's counters
    if (et == 0) ticket = atom_add_acq_rel_gpu(&p.hdr->done, 1u);
    // Hand an accumulator buffer back to the MMA thread (the leader's, for
    // a CTA pair).
    auto release_acc = [&](int b) {
      if constexpr (C::PAIR) mbar_arrive_cluster(cluster_addr(&tempty_bar[b], 0));
      else mbar_arrive(&tempty_bar[b]);
    };

    Cursor cur;
    cur.init(s, unit);
    Work w;
    int ab = 0;
    uint32_t aphase = 0;
    int bsel = 0;
    uint32_t c0_phase = 0;     // bit b: parity of the next C0 copy into staging buffer b
    bool c0r_pending = false;  // C0 copies into the ring not yet waited for
    int estage = 0;            // in-CTA ABFT: the epilogue's place in the stage ring
    uint32_t ephase = 0;
    int xpar = 0;              // ILC pairs: exchange slot (and barrier parity) of the next tile
    int nseg = 0;
    bool store_ok = true;
    bool ck_ready = false;
    if (enc_here) {
      // Encode pass (bf16): column sums of each unit's boxes out of the ring,
      // then the unit's hi / lo encoding rows and its max |element|.
      int u0, u1;
      enc_in_units(p, (int)blockIdx.x - s.g, s.g_ck, u0, u1);
      const int units_a = p.enc_tiles_a * p.enc_slices;
      float* part = reinterpret_cast<float*>(epi);  // [4 warps][256 columns]
      int est = 0;
      uint32_t eph = 0;
      bool eok = true;
      for (int u = u0; u < u1 && eok; ++u) {
        const bool is_a = u < units_a;
        const int t = u / p.enc_slices, sl = u - t * p.enc_slices;
        const int nsub = is_a ? kBM / kEncInRows : p.enc_bn / kEncInRows;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        float amax = 0.f;
        for (int h = 0; h < nsub; ++h) {
          const bool got = wait_bar(&full_bar[est], eph, aux, limit);
          if (!got && !aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
          if (!epi_all(got && !aborted(aux))) {
            eok = false;
            break;
          }
          // Warp ew sums rows ew, ew + 4, ...; lane l holds columns 8l .. 8l + 7.
          const uint8_t* st = ring + est * C::STAGE_BYTES + lane * 16;
#pragma unroll 4
          for (int i = 0; i < kEncInRows / 4; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(st + (ew + 4 * i) * (kEncInCols * 2));
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = __uint_as_float(wv[j] << 16);
              const float hi = __uint_as_float(wv[j] & 0xffff0000u);
              acc[2 * j] += lo;
              acc[2 * j + 1] += hi;
              amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
            }
          }
          named_bar_sync(1, kEpiThreads);  // the stage is read
          if (et == 0) mbar_arrive(&empty_bar[est]);
          if (++est == STAGES) {
            est = 0;
            eph ^= 1;
          }
        }
        if (!eok) break;
#pragma unroll
        for (int i = 0; i < 8; ++i) part[ew * kEncInCols + lane * 8 + i] = acc[i];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) aux->tmax_a[ew] = amax;
        named_bar_sync(1, kEpiThreads);
        __nv_bfloat16* enc = static_cast<__nv_bfloat16*>(is_a ? p.enc_a_w : p.enc_b_w);
        const int tile = is_a ? t : t - p.enc_tiles_a;
        __nv_bfloat16* hi_row = enc + (int64_t)(kEncRows * tile) * p.enc_kp;
        __nv_bfloat16* lo_row = hi_row + p.enc_kp;
#pragma unroll
        for (int hh = 0; hh < kEncInCols / kEpiThreads; ++hh) {
          const int c = hh * kEpiThreads + et;
          const float x = part[c] + part[kEncInCols + c] + part[2 * kEncInCols + c] +
                          part[3 * kEncInCols + c];
          const int col = sl * kEncInCols + c;
          if (col < p.enc_kp) {  // columns in [k, kp) hold zero sums
            const __nv_bfloat16 hv = __float2bfloat16_rn(x);
            hi_row[col] = hv;
            lo_row[col] = __float2bfloat16_rn(x - __bfloat162float(hv));
          }
        }
        if (et == 0) {
          p.umax_w[u] = fmaxf(fmaxf(aux->tmax_a[0], aux->tmax_a[1]),
                              fmaxf(aux->tmax_a[2], aux->tmax_a[3]));
          if (sl == 0) p.pub_w[t].scale_exp = 0;
        }
        named_bar_sync(1, kEpiThreads);  // part and tmax reused by the next unit
      }
      // The checksum segments add into cr_all / ccT_all: this CTA zeroes its
      // share of them first.
      if (p.ck_atomic) {
        const int64_t ncr = (int64_t)p.m * p.ld_cr / 4, ncc = (int64_t)p.n * p.ld_cc / 4;
        const int j = (int)blockIdx.x - s.g;
        float4* zcr = reinterpret_cast<float4*>(const_cast<float*>(p.cr_all));
        float4* zcc = reinterpret_cast<float4*>(const_cast<float*>(p.cc_all));
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t i = j * (int64_t)kEpiThreads + et; i < ncr; i += (int64_t)s.g_ck * kEpiThreads)
          zcr[i] = z;
        for (int64_t i = j * (int64_t)kEpiThreads + et; i < ncc; i += (int64_t)s.g_ck * kEpiThreads)
          zcc[i] = z;
      }
      // Every encode write of this CTA lands before the counter moves.
      __threadfence();
      named_bar_sync(1, kEpiThreads);
      if (et == 0 && eok) {
        __threadfence();
        atomicAdd(&p.hdr->enc_done[par], 1u);
      }
    }
    while (cur.next(s, w)) {
      if (p.trace && et == 0) {
        int32_t* tr = p.trace + (size_t)blockIdx.x * SKG_TRACE_STRIDE;
        if (nseg < SKG_TRACE_CAP) {
          tr[1 + 4 * nseg] = w.tile - s.t_ck;
          tr[2 + 4 * nseg] = w.kb_begin;
          tr[3 + 4 * nseg] = w.kb_end;
          tr[4 + 4 * nseg] = w.role;
        }
        tr[0] = nseg + 1;
      }
      ++nseg;
      const bool is_ck = w.tile < s.t_ck;  // a fused checksum-GEMM tile
      // The CTA's last work item: once its accumulator is full, no copy or
      // MMA touches the stage ring again.
      bool last_item;
      {
        Cursor peek = cur;
        Work wn;
        last_item = !peek.next(s, wn);
      }
      int tm = 0, tn = 0;
      if (!is_ck) tile_coords(s, w.tile, tm, tn);
      // This CTA's 128-row tile: a pair tile is two of them.
      if (C::PAIR) tm = 2 * tm + (int)crank;
      const int m0 = tm * kBM;
      const int n0 = tn * BN;
      // beta != 0: pull this warp's rows of C0 into L2 while the mainloop
      // runs, so the epilogue's C0 loads do not wait on DRAM.
      if (p.beta != 0.f && !is_ck && w.role != kRolePeer && lane == 0 && m0 + q * 32 < p.m) {
#pragma unroll 1
        for (int c = 0; c < BN / C::EPI_COLS && n0 + c * C::EPI_COLS < p.n; ++c)
          tma_prefetch_l2_2d(&tmC, n0 + c * C::EPI_COLS, m0 + q * 32);
      }

      // Inputs of this tile's ABFT check that do not depend on its
      // accumulator (the encode pass's maxima and scales, the reference
      // checksums): their loads are issued before the accumulator wait and
      // first used after it, so their latency hides behind the mainloop.
      float pf_ma = 0.f, pf_mb = 0.f, pf_cr0 = 0.f, pf_cr1 = 0.f;
      float pf_cc0[C::CC_GROUPS], pf_cc1[C::CC_GROUPS];
#pragma unroll
      for (int h = 0; h < C::CC_GROUPS; ++h) pf_cc0[h] = pf_cc1[h] = 0.f;
      int pf_ea = 0, pf_eb = 0;
      // (A CTA pair's second half lies past m when m has an odd number of
      // 128-row tiles: nothing there to check.)
      const bool verify_here = C::ABFT && !is_ck && w.role != kRolePeer && m0 < p.m;
      if constexpr (C::LOCAL) {
        // Reference checksums formed here from the shared-memory stages
        // while the MMAs run (one whole tile per CTA).
        float* scratch = reinterpret_cast<float*>(epi);
        const int nk = w.kb_end - w.kb_begin;
        const LocalSums<BN> ls =
            p.in_f16 ? local_checksums<C, true>(p, ring, full_bar, empty_bar, estage, ephase, nk,
                                                scratch, ew, lane, et, r, aux, limit)
                     : local_checksums<C, false>(p, ring, full_bar, empty_bar, estage, ephase, nk,
                                                 scratch, ew, lane, et, r, aux, limit);
        if (!ls.ok) break;
        estage = ls.stage;
        ephase = ls.phase;
        pf_cr0 = ls.cr;
#pragma unroll
        for (int h = 0; h < C::CC_GROUPS; ++h) pf_cc0[h] = ls.cc[h];
        pf_ma = ls.ma;
        pf_mb = ls.mb;
      }
      // A tile whose references come late -- the first output tile of a
      // launch whose side CTAs run the encode pass, since they store the
      // references only once every one of them has encoded and added its
      // checksum rows -- with beta = 0 and no fixup is stored first and
      // checked once the references are in; a located fault then has its
      // corrected value written over the element (the accumulator stays in
      // TMEM until the check).
      // (Only the launches that run the encode pass in their side CTAs can
      // have such tiles: 128-wide tiles on single CTAs.)
      constexpr bool kStoreFirst =
          C::ABFT && !C::PAIR && !C::LOCAL && !C::ILC && !C::MN && BN == 128;
      const bool spec = kStoreFirst && verify_here && w.role == kRoleFull && p.beta == 0.f &&
                        p.ck_atomic && s.t_ck > 0 && !ck_ready;
      // Wait until the fused checksum tiles are all stored (false: timed out).
      auto wait_references = [&]() -> bool {
        // The fused checksum tiles must all be stored first. Every CTA runs
        // its own share of them before its first output tile, and dedicated
        // checksum CTAs wait only for each other (all resident), so this
        // wait ends.
        bool fine = true;
        if (et == 0) {
          const uint64_t t0 = globaltimer();
          const uint32_t ck_want =
              p.ck_atomic ? (uint32_t)p.ck_target : (uint32_t)(kCkHalf * s.t_ck);
          while (ld_acquire_gpu(&p.hdr->ck_done[par]) < ck_want) {
            nanosleep_ns(128);
            if (globaltimer() - t0 > limit) {
              record_error(p, aux, SKG_ERR_FIXUP_TIMEOUT);
              fine = false;
              break;
            }
          }
        }
        return epi_all(fine && !aborted(aux));
      };
      // Loads of the references and of the thresholds' inputs (pf_*).
      auto load_references = [&]() {
        const float* ua = p.umax + (int64_t)tm * p.enc_slices;
        const float* ub = p.umax + (int64_t)(p.enc_tiles_a + tn) * p.enc_slices;
        if (et < p.enc_slices) {
          pf_ma = __ldcg(ua + et);
          pf_mb = __ldcg(ub + et);
        }
        pf_ea = p.pub_a[tm].scale_exp;
        pf_eb = p.pub_b[tn].scale_exp;
        if (!C::ILC && m0 + r < p.m) {
          const float* crp = p.cr_all + (int64_t)(m0 + r) * p.ld_cr + kEncRows * tn;
          pf_cr0 = __ldcg(crp);
          pf_cr1 = __ldcg(crp + 1);
        }
#pragma unroll
        for (int h = 0; h < C::CC_GROUPS; ++h) {
          const int col = n0 + h * 128 + r;
          if (!C::ILC && col < p.n) {
            const float* ccp = p.cc_all + (int64_t)col * p.ld_cc + kEncRows * tm;
            pf_cc0[h] = __ldcg(ccp);
            pf_cc1[h] = __ldcg(ccp + 1);
          }
        }
        // More encode units than epilogue threads (k above 128 slices).
        for (int j = et + kEpiThreads; j < p.enc_slices; j += kEpiThreads) {
          pf_ma = fmaxf(pf_ma, __ldcg(ua + j));
          pf_mb = fmaxf(pf_mb, __ldcg(ub + j));
        }
      };
      if (!C::LOCAL && verify_here && !spec) {
        if (!C::ILC && s.t_ck > 0 && !ck_ready) {
          if (!wait_references()) break;
          ck_ready = true;
        }
        load_references();
      }

      // Mid-mainloop fault injection (testing only): once the MMAs up to MAC
      // iteration inj_kb are done, the warp of the row's lane quadrant flips
      // the value in TMEM and releases the MMA thread (kept out of line).
      if (p.inj_kb >= 0 && mid_inject_item<C::PAIR>(p, s, w, (int)crank) &&
          q == (p.inj_row[0] >> 5))
        mid_inject_flip<C::PAIR>(p, tmem_base + ab * C::ACC_COLS, q, lane, inj_bar, injdone_bar,
                                 aux, limit);

      bool got = wait_bar_inline<C::PAIR>(&tfull_bar[ab], aphase, aux, limit);
      if (!got && !aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
      if (!epi_all(got && store_ok && !aborted(aux))) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + ab * C::ACC_COLS + ((uint32_t)(q * 32) << 16);
      const int out_tile = tm * s.tiles_n + tn;  // row-major 128 x BLK_N tile number
      if constexpr (C::ILC) {
        if (!is_ck) {
          // The reference checksums the MMAs accumulated next to the tile:
          // row r's cr (hi, lo) and, in lane r, the cc of B row r.
          uint32_t u[32];
          tmem_ld32(tacc + C::CR_COL, u);
          pf_cr0 = f32_of(u[0]);
          pf_cr1 = f32_of(u[1]);
          if constexpr (!C::PAIR) {
            pf_cc0[0] = f32_of(u[16]);
            pf_cc1[0] = f32_of(u[17]);
          } else {
            // Lane r of CTA c holds B row c * 128 + r: its column sums for
            // this half's e^T A (cols 16 + 8c) and for the other half's
            // (16 + 8 (1 - c)). The halves swap the latter through xbuf.
            const float s0 = f32_of(u[16]) + f32_of(u[17]);  // for half 0's e^T A
            const float s1 = f32_of(u[24]) + f32_of(u[25]);  // for half 1's e^T A
            const float mine = crank == 0 ? s0 : s1, theirs = crank == 0 ? s1 : s0;
            float* slot = xbuf + xpar * 128 + r;
            st_shared_cluster_f32(cluster_addr(slot, 1u - crank), theirs);
            mbar_arrive_cluster(cluster_addr(xch_bar, 1u - crank));
            const bool got_x = wait_bar(xch_bar, (uint32_t)xpar, aux, limit, true, true);
            if (!got_x && !aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
            const float peer = got_x ? *reinterpret_cast<volatile float*>(slot) : 0.f;
            // columns h * 128 + r: h = crank from this CTA, the other from the peer
            pf_cc0[0] = crank == 0 ? mine : peer;
            pf_cc0[1] = crank == 0 ? peer : mine;
            pf_cc1[0] = pf_cc1[1] = 0.f;
            xpar ^= 1;  // next tile: the other slot and barrier phase parity
          }
        }
      }
      // Fault injection (testing only): this tile gets a flip after its fixup.
      // Split reduction (see Schedule::split_max): this CTA is one of the
      // parts that finish the tile, each storing a range of its columns.
      constexpr int kChunks = BN / C::EPI_COLS;
      // (Single CTAs only: the pair kernels have no registers to spare.)
      const bool split = !C::ABFT && !C::PAIR && !is_ck && Cursor::split(s, w) &&
                         unit <= w.part_last && w.share_parts <= kChunks;
      const bool inject_here = !is_ck && (w.role != kRolePeer || split) &&
                               ((out_tile == p.inj_tile[0] && p.inj_kb < 0) ||
                                out_tile == p.inj_tile[1]);
      // ... or got one in the mainloop (fault records say "injected").
      const bool injected_tile =
          !is_ck && (out_tile == p.inj_tile[0] || out_tile == p.inj_tile[1]);
      // This segment's region of fixup storage (flags at a fixed place).
      uint32_t* rflags = p.flags + (size_t)w.region * kMaxCtas;
      float* rpartials = p.partials + (size_t)w.region * p.ws_ctas * kBM * BN;
      float* my_slot = rpartials + (size_t)my_slot_idx * kBM * BN;
      // Columns of the accumulator that carry data: a checksum tile uses
      // only its first ck_n_* columns.
      const int live_chunks =
          !is_ck ? BN / 32
                 : ((w.tile < p.ck_cr_tiles ? p.ck_n_cr : p.ck_n_cc) + 31) / 32;

      // Shared reduction of a tile that at least share_min CTAs end in (all
      // of them store partials, the owner too; see reduce_share). An owner
      // whose range began in an earlier tile keeps this partial and its flag
      // in bank 2 (the second region's storage), since its slot holds the
      // earlier tile's partial.
      const bool share = !C::ABFT && Cursor::shared(s, w) && unit <= w.part_last;
      // A split part `sj` of `sp` finishes the tile's column chunks [c_lo, c_hi).
      int c_lo = 0, c_hi = kChunks;
      if (split) {
        const int sp = w.share_parts, sj = unit - w.owner;
        c_lo = sj * kChunks / sp;
        c_hi = (sj + 1) * kChunks / sp;
      }
      if ((share || split) && w.role == kRoleOwner && w.owner_bank2) {
        rflags += kMaxCtas;
        my_slot += (size_t)p.ws_ctas * kBM * BN;
      }
      // StorePartials + Signal (Algorithm 5, non-started segment): peers,
      // the parts of a shared reduction, and the parts of a split one (which
      // keep the accumulator for their own columns).
      // (Checksum-tile segments that add into the reference arrays store no
      // partial and wait for no peer.)
      const bool ck_add = C::ABFT && is_ck && p.ck_atomic;
      const bool stores_partial = (w.role == kRolePeer && !ck_add) || share || split;
      if (stores_partial) {
#pragma unroll 1
        for (int c32 = 0; c32 < live_chunks; ++c32) {
          uint32_t u[32];
          tmem_ld32(tacc + c32 * 32, u);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_cg_f4(partial_at<BN>(my_slot, c32 * 8 + j, r, w.region == 0),
                     make_float4(f32_of(u[4 * j]), f32_of(u[4 * j + 1]), f32_of(u[4 * j + 2]),
                                 f32_of(u[4 * j + 3])));
        }
        if (!split) {
          tc_fence_before();
          release_acc(ab);
        }
        named_bar_sync(1, kEpiThreads);
        if (et == 0 && (int)blockIdx.x != p.drop_signal) {
          __threadfence();
          st_release_gpu(&rflags[my_slot_idx], epoch);
        }
        if (share && !reduce_share<C>(p, rpartials, p.flags, w.owner, w.owner_bank2,
                                      w.contrib_last, w.part_last, unit, slot_stride, (int)crank,
                                      m0, n0, ew, lane, epoch, out_tile, aux, limit))
          break;
      }
      if (!stores_partial || split) {
        const bool owner = (w.role == kRoleOwner);
        if ((owner && !ck_add) || split) {
          // Wait for every other CTA that covers part of this tile (an
          // owner: the later ones; a split part: all of them, the owner's
          // flag in bank 2 when it began earlier): the lanes of one warp
          // poll up to 32 flags at once.
          const int first_cover = split ? w.owner : unit + 1;
          const int last_cover = split ? w.contrib_last : w.peer_last;
          bool fine = true;
          if (ew == 0) {
            for (int peer = first_cover + lane; peer <= last_cover && fine; peer += 32) {
              if (peer == unit) continue;
              const int fi = peer * slot_stride + (int)crank +
                             (split && peer == w.owner && w.owner_bank2 ? kMaxCtas : 0);
              const uint32_t* pf = split ? p.flags : rflags;
              if (ld_acquire_gpu(&pf[fi]) == epoch) continue;
              if (ld_acquire_gpu(&rflags[fi]) == epoch) continue;
              const uint64_t t0 = globaltimer();
              uint32_t spins = 0;
              while (ld_acquire_gpu(&pf[fi]) != epoch) {
                if (++spins > 64) nanosleep_ns(64);
                if ((spins & 15) == 0 && globaltimer() - t0 > limit) {
                  record_error(p, aux, SKG_ERR_FIXUP_TIMEOUT);
                  fine = false;
                  break;
                }
              }
            }
          }
          if (!epi_all(fine && !aborted(aux))) {
            tc_fence_before();
            release_acc(ab);
            break;
          }
        }
        // The CTA's last output tile: once its accumulator is full the stage
        // ring is idle, so each epilogue warp takes a quarter of it and
        // fetches what its 32 rows still need with bulk copies in flight
        // together, rather than one round trip per 32-column chunk:
        //  - beta != 0: the quadrant's rows of C0, read by the store pass;
        //  - LoadPartials (owner): every peer's band of this quadrant, in
        //    half-band pieces through a few pipelined slots, folded into the
        //    accumulator in TMEM, so the passes below see it fixed up.
        // (Runs at most once per CTA, so the barrier parities start at 0.)
        bool add_partials = owner && !split;
        bool c0_ring = false;
        constexpr uint32_t kQuarter = (uint32_t)(STAGES * C::STAGE_BYTES / 4) & ~1023u;
        constexpr uint32_t kC0Bytes = 32u * BN * C::OUT_BYTES;
        constexpr uint32_t kC0Off = (kQuarter - kC0Bytes) & ~1023u;
        constexpr uint32_t kHalf = kPartialBandBytes<BN> / 2;
        // (ILC launches split no tile, so they have no owner fixup to fit.)
        static_assert(kC0Bytes <= kQuarter && (C::ILC || kC0Off >= kHalf),
                      "ring quarter too small");
        uint8_t* qring = ring + ew * kQuarter;
        if (last_item && !is_ck && (w.role != kRolePeer || split)) {
          c0_ring = p.beta != 0.f && m0 + q * 32 < p.m;  // warp-uniform
          if (c0_ring && lane == 0) {
            int nbox = c_lo;
            while (nbox < c_hi && n0 + nbox * C::EPI_COLS < p.n) ++nbox;
            mbar_arrive_expect_tx(&c0r_bar[ew], (uint32_t)(nbox - c_lo) * C::EPI_BUF_BYTES);
            for (int c = c_lo; c < nbox; ++c)
              tma_load_2d(qring + kC0Off + c * C::EPI_BUF_BYTES, &tmC, &c0r_bar[ew],
                          n0 + c * C::EPI_COLS, m0 + q * 32);
          }
          c0r_pending = c0_ring;
        }
        if (split) {
          const uint32_t room = c0_ring ? kC0Off : kQuarter;
          const int slots = min(kFixSlots, (int)(room / kHalf));
          const bool fine = fold_split_through_ring<BN>(
              qring, slots, rpartials, (size_t)p.ws_ctas * kBM * BN, w.owner, w.owner_bank2,
              w.contrib_last, unit, slot_stride, (int)crank, q, lane, tacc, c_lo * C::EPI_COLS,
              c_hi * C::EPI_COLS, &fix_bar[ew * kFixSlots], p, aux, limit);
          if (!epi_all(fine && !aborted(aux))) {
            tc_fence_before();
            release_acc(ab);
            break;
          }
        } else if (!C::ILC && owner && !is_ck && last_item) {
          const uint32_t room = c0_ring ? kC0Off : kQuarter;
          const int slots = min(kFixSlots, (int)(room / kHalf));
          const bool fine = fixup_through_ring<BN>(
              qring, slots, rpartials, unit, w.peer_last, slot_stride, (int)crank, q, lane, tacc,
              &fix_bar[ew * kFixSlots], p, aux, limit);
          if (!epi_all(fine && !aborted(aux))) {
            tc_fence_before();
            release_acc(ab);
            break;
          }
          add_partials = false;
        }

        if (C::ABFT && is_ck) {
          // -------------------------------------------- fused checksum tile
          // Store fp32 rows of cr_all or ccT_all (ck_atomic: add this
          // segment's rows into them), then count the tile (segment) done
          // once every warp's stores have landed.
          const bool cr_side = w.tile < p.ck_cr_tiles;
          const CUtensorMap* mapC = cr_side ? &tmCr : &tmCc;
          const int rows = cr_side ? p.m : p.n;
          const int ncols = cr_side ? p.ck_n_cr : p.ck_n_cc;
          const int r0 = ((cr_side ? w.tile : w.tile - p.ck_cr_tiles) * kCkHalf + (int)crank) * kBM;
          const int nchunks = (ncols + 31) / 32;
          const bool live = (r0 + q * 32) < rows;
#pragma unroll 1
          for (int c = 0; c < nchunks; ++c) {
            uint32_t u[32];
            float v[32];
            tmem_ld32(tacc + c * 32, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = f32_of(u[i]);
            if (owner && !ck_add)
              add_peer_partials<BN>(v, rpartials, unit + 1, w.peer_last, c, r, w.region == 0,
                                    slot_stride, (int)crank);
            if (c == nchunks - 1) {
              tc_fence_before();
              release_acc(ab);
            }
            if (!live || !store_ok) continue;  // warp-uniform
            uint8_t* buf = ebuf + bsel * C::EPI_BUF_BYTES;
            if (lane == 0) bulk_wait_read<C::EPI_BUFS - 1>();
            __syncwarp();
            uint32_t wv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) wv[i] = __float_as_uint(v[i]);
            staging_write(buf, lane, wv);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (ck_add) tma_reduce_add_2d(mapC, buf, c * 32, r0 + q * 32);
              else tma_store_2d(mapC, buf, c * 32, r0 + q * 32);
              bulk_commit();
            }
            bsel = (bsel + 1) % C::EPI_BUFS;
          }
          if (lane == 0) bulk_wait<0>();
          __syncwarp();
          named_bar_sync(1, kEpiThreads);
          if (et == 0) {
            __threadfence();
            atomicAdd(&p.hdr->ck_done[par], 1u);
          }
          if (++ab == ACC_BUFS) {
            ab = 0;
            aphase ^= 1;
          }
          continue;
        }

        // ------------------------------------------------ ABFT verify
        int fix_row = -1, fix_col = -1;
        float fix_val = 0.f;
        auto check = [&](bool flips) {
          const TileFix f = check_tile<C>(
              p, aux, epi, tacc, q, lane, et, r, add_partials, rpartials, unit, w.peer_last,
              w.region == 0, slot_stride, (int)crank, inject_here, flips, injected_tile, out_tile,
              epoch, pf_ma, pf_mb, pf_cr0, pf_cr1, pf_cc0, pf_cc1, pf_ea, pf_eb);
          fix_row = f.row;
          fix_col = f.col;
          fix_val = f.val;
        };
        if (verify_here && !spec) check(true);
        if (kStoreFirst && spec && inject_here) {
          // Testing flips land in TMEM before the tile is stored.
#pragma unroll 1
          for (int c32 = 0; c32 < BN / 32; ++c32) {
            uint32_t u[32];
            tmem_ld32(tacc + c32 * 32, u);
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = f32_of(u[i]);
            float clean = 0.f;
            const bool hit = apply_flips(p, out_tile, r, c32, v, &clean);
            if (hit) aux->inj_clean = clean;
            if (__any_sync(0xffffffffu, hit)) {
              uint32_t wv[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) wv[i] = __float_as_uint(v[i]);
              tmem_st32(tacc + c32 * 32, wv);
            }
          }
        }

        // ------------------------------------------------ StoreTile
        const bool rows_live = (m0 + q * 32) < p.m;
        // beta != 0 outside the ring: each chunk's C0 rows come through its
        // staging buffer, and the next chunk's copy is issued into the other
        // buffer as soon as this chunk's rows are in registers, so the round
        // trips overlap the combine and store of the chunk before.
        const bool c0_staged = p.beta != 0.f && !c0_ring;
        static_assert(C::EPI_BUFS == 2, "two C0 barriers per epilogue warp");
        bool c0_ahead = false;  // this chunk's C0 copy is already in flight
#pragma unroll 1
        for (int c = c_lo; c < c_hi; ++c) {
          const int col0 = n0 + c * C::EPI_COLS;
          const bool st_chunk = rows_live && col0 < p.n && store_ok;  // warp-uniform
          uint8_t* buf = ebuf + bsel * C::EPI_BUF_BYTES;
          if (st_chunk && !c0_ahead) {
            // Free the staging buffer and start its C0 load before the
            // accumulator columns are read, so the latencies overlap.
            if (lane == 0) bulk_wait_read<C::EPI_BUFS - 1>();
            __syncwarp();
            if (c0_staged && lane == 0) {
              mbar_arrive_expect_tx(&c0_bar[2 * ew + bsel], C::EPI_BUF_BYTES);
              tma_load_2d(buf, &tmC, &c0_bar[2 * ew + bsel], col0, m0 + q * 32);
            }
          }
          c0_ahead = false;
          float y[C::EPI_COLS];
#pragma unroll
          for (int hh = 0; hh < C::EPI_COLS / 32; ++hh) {
            uint32_t u[32];
            const int c32 = c * (C::EPI_COLS / 32) + hh;
            float v[32];
            tmem_ld32(tacc + c32 * 32, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = f32_of(u[i]);
            if (!C::ABFT && add_partials)
              add_peer_partials<BN>(v, rpartials, unit + 1, w.peer_last, c32, r, w.region == 0,
                                    slot_stride, (int)crank);
#pragma unroll
            for (int i = 0; i < 32; ++i) y[hh * 32 + i] = v[i];
            if (!C::ABFT) {
              if (inject_here && apply_flips(p, out_tile, r, c32, v, nullptr)) {
#pragma unroll
                for (int i = 0; i < 32; ++i) y[hh * 32 + i] = v[i];
              }
            } else if (r == fix_row && (fix_col >> 5) == c32) {
              const int jc = fix_col & 31;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i == jc) y[hh * 32 + i] = fix_val;
            }
          }
          if (c == c_hi - 1 && !spec) {
            // Accumulator fully read: hand the TMEM buffer back to the MMA warp.
            tc_fence_before();
            release_acc(ab);
          }
          if (!st_chunk) continue;
          if (p.beta != 0.f) {
            const uint8_t* c0src = buf;
            bool got_c0;
            if (c0_ring) {
              got_c0 = !c0r_pending ||
                       __all_sync(0xffffffffu, wait_bar(&c0r_bar[ew], 0, aux, limit));
              if (got_c0) c0r_pending = false;
              c0src = qring + kC0Off + c * C::EPI_BUF_BYTES;
            } else {
              got_c0 = __all_sync(0xffffffffu, wait_bar(&c0_bar[2 * ew + bsel],
                                                        (c0_phase >> bsel) & 1u, aux, limit));
            }
            if (!got_c0) {
              if (lane == 0 && !aborted(aux)) record_error(p, aux, SKG_ERR_PIPELINE_TIMEOUT);
              store_ok = false;  // stop storing; the next tile boundary exits
              continue;
            }
            if (!c0_ring) c0_phase ^= 1u << bsel;
            uint32_t w0[32];
            staging_read(c0src, lane, w0);
            const int cn = c + 1;
            if (c0_staged && cn < c_hi && n0 + cn * C::EPI_COLS < p.n) {
              // The next buffer last held the previous chunk's output: once
              // that store has read it, it takes the next chunk's C0 rows.
              const int nb = (bsel + 1) % C::EPI_BUFS;
              if (lane == 0) {
                bulk_wait_read<C::EPI_BUFS - 2>();
                mbar_arrive_expect_tx(&c0_bar[2 * ew + nb], C::EPI_BUF_BYTES);
                tma_load_2d(ebuf + nb * C::EPI_BUF_BYTES, &tmC, &c0_bar[2 * ew + nb],
                            n0 + cn * C::EPI_COLS, m0 + q * 32);
              }
              c0_ahead = true;
            }
            float c0v[C::EPI_COLS];
            unpack_row<C::OUT>(w0, c0v);
#pragma unroll
            for (int i = 0; i < C::EPI_COLS; ++i) y[i] = p.alpha * y[i] + p.beta * c0v[i];
          } else {
#pragma unroll
            for (int i = 0; i < C::EPI_COLS; ++i) y[i] = p.alpha * y[i];
          }
          uint32_t wout[32];
          pack_row<C::OUT>(y, wout);
          staging_write(buf, lane, wout);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, buf, col0, m0 + q * 32);
            bulk_commit();
          }
          bsel = (bsel + 1) % C::EPI_BUFS;
        }
        if (kStoreFirst && spec) {
          // Stored before its check: the references are in once every
          // checksum segment has been added; check the tile against them.
          const bool fine = wait_references();
          if (fine) {
            ck_ready = true;
            load_references();
            check(false);
            if (fix_row >= 0 && q == (fix_row >> 5) && store_ok) {
              // The located element was stored from the faulty accumulator:
              // once this warp's tile stores have landed, the corrected
              // value goes over it (beta = 0: C = alpha acc).
              if (lane == 0) bulk_wait<0>();
              __syncwarp();
              if (r == fix_row && m0 + r < p.m && n0 + fix_col < p.n) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                store_out<C::OUT>(p.c_ptr, (int64_t)(m0 + r) * p.ldc + n0 + fix_col,
                                  p.alpha * fix_val);
              }
            }
          }
          tc_fence_before();
          release_acc(ab);
          if (!fine) break;
        }
      }
      if (++ab == ACC_BUFS) {
        ab = 0;
        aphase ^= 1;
      }
    }
    // C0 copies into the ring that an early exit left unwaited land before
    // the CTA leaves; output stores only need to have read their staging
    // (the grid's completion makes the writes visible to later work).
    if (c0r_pending && lane == 0) wait_bar(&c0r_bar[ew], 0, aux, limit, false);
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (C::PAIR) {
    // A peer's copies complete on the leader's barriers, so after an abort
    // this CTA cannot see its own copies land: give them time before the
    // pair parts. Then neither CTA leaves while the other may still signal
    // its barriers or read its shared memory.
    if (aborted(aux)) {
      const uint64_t t0 = globaltimer();
      while (globaltimer() - t0 < 100000) nanosleep_ns(1000);
    }
    cluster_sync();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (C::PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  // The CTA with the launch's last ticket (every CTA took one after reading
  // the epoch) readies the workspace for the next launch: tickets back to
  // zero, the next parity's counters cleared, the epoch advanced.
  if (threadIdx.x == 64) {  // epilogue thread 0, which holds the ticket
    if (p.cta_clock) p.cta_clock[2 * blockIdx.x + 1] = globaltimer();
    if (ticket == gridDim.x - 1) {
      const uint32_t e = aux->epoch - 1u;
      p.hdr->done = 0;
      p.hdr->ck_done[(e + 1u) & 1u] = 0;
      p.hdr->enc_done[(e + 1u) & 1u] = 0;
      atomicAdd(&p.report->launches, 1u);
      st_release_gpu(&p.hdr->epoch, e + 1u);
    }
  }
}

}  // namespace skg
