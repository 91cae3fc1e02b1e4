// C-ABI entry points of libskgemm.so (declared in include/skgemm.h).
//
// Host side of one gemm call: validate the BLAS-style arguments (the
// problem statement C = alpha A B + beta C of "Stream-K: Work-centric
// Parallel Decomposition for Dense Matrix-Matrix Multiplication on the GPU",
// §A3), choose BLK_N and the grid, lay out the caller's workspace, encode the
// TMA descriptors, run the ABFT encode pass when asked, and launch the
// persistent kernel. Nothing here computes any part of the product.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "skg_internal.h"
#include "skg_model.h"
#include "skgemm.h"

using namespace skg;

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr size_t kHeaderBytes = 8192;  // WsHeader + skg_report_t, rounded

static_assert(256 + sizeof(skg_report_t) <= kHeaderBytes, "report does not fit the header");

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

int sm_count_cached() {
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && counts[dev] > 0) return counts[dev];
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev < 64) counts[dev] = v;
  return v;
}

// The library does not pick in-CTA ABFT references by itself: on GB300 the
// four epilogue warps (one per SM sub-partition, little latency hiding)
// take ~1.5 us per 128 x 128 x 64 k-step for the sums, several times the
// MMA's time, so a 1024^3 call took 35 us against 23 us on the fused
// checksum path. skg_opts_t.abft_local = 2 selects them.

struct Resolved {
  int sched;
  int grid;     // CTAs launched for the output tiles (two per cluster with pairs)
  int pair;     // 1: clusters of two CTAs, 256 x BLK_N tiles, one M = 256 MMA
  int grid_max; // CTAs that can be resident (pairs: two per resident cluster)
  int grid_ck;  // dedicated side CTAs launched after the grid ones
  int grid_ckt; // of those, the ones that run checksum tiles (the rest only encode)
  int bn;
  int abft;
  float tau_row, tau_col;
  int inj_tile[2], inj_row[2], inj_col[2], inj_bit[2];  // testing: up to two flips
  int inj_kb;   // >= 0: flip 0 inside the mainloop after this MAC iteration
  int stagger;  // StaggerU-style k staggering (> 1 = on)
  uint64_t timeout_ns;
  int32_t* trace;
  uint64_t* cta_clock;
  int drop_signal;
  int preencoded;
  int raster_band;
  int enc_inkernel;  // the dedicated side CTAs run the encode pass (no encode launch)
  int abft_local;    // ABFT references formed in each CTA (one whole tile per CTA)
  int ilc;           // ABFT references accumulated by the output tiles' MMAs (DP plan)
  int ws_grid;
  int64_t k_for_plan;  // CTAs the workspace's flags and partial slots are sized for
  // Shared reduction of the output Stream-K tiles (no ABFT): Schedule's
  // share_min and share_bank2 (bank 2 takes the second region's storage).
  int share_min;
  int share_bank2;
  int split;  // split reduction of the output tiles (Schedule::split_max)
  int ck_atomic;  // checksum-tile segments add into zeroed references (KernelParams)
};

// Whether an ABFT call runs its reference checksums inside the mainloop
// (skg_opts_t.abft_inloop): always when asked, never when refused; left to
// the library, for shapes whose data-parallel plan needs at most two waves
// of tiles, where the separate checksum tiles' chain of global
// synchronisations is longer than the mainloop (measured on GB300).
bool ilc_wanted(int64_t m, int64_t n, int64_t k, const skg_opts_t* o, const Resolved& r,
                int ms) {
  if (o->abft_inloop == 1) return false;
  if (o->abft_inloop == 2) return true;
  return false;
}

// Schedule, g and BLK_N: whatever the options leave open is chosen by the
// grid-size model (skg_model.h). A fixed schedule with grid 0 runs on all
// SMs, as the page's persistent launches do.
skg_status_t resolve(int64_t m, int64_t n, int64_t k, const skg_opts_t* o, Resolved& r,
                     int sms, bool compact = false) {
  skg_opts_t d;
  skg_opts_default(&d);
  if (!o) o = &d;
  if (o->sched < SKG_SCHED_DP || o->sched > SKG_SCHED_AUTO) return SKG_ERR_ARG;
  if (o->tile_n != 0 && o->tile_n != 64 && o->tile_n != 128 && o->tile_n != 256)
    return SKG_ERR_UNSUPPORTED;
  // 64-wide tiles: GEMMs without ABFT on single CTAs.
  if (o->tile_n == 64 && (o->abft || o->cta_pair == 2)) return SKG_ERR_UNSUPPORTED;
  if (o->grid < 0) return SKG_ERR_ARG;
  const int ms = sms > 0 ? sms : 256;  // no device: plan for a large part
  if (o->grid > 0 && sms > 0 && o->grid > sms) return SKG_ERR_UNSUPPORTED;  // co-residency
  r.abft = o->abft ? 1 : 0;
  const int want_sched = o->sched == SKG_SCHED_AUTO ? -1 : o->sched;
  const int want_grid = o->grid > 0 ? o->grid : (want_sched >= 0 ? ms : 0);
  // Launches without ABFT reduce shared tiles together (the model knows).
  const bool share = !o->abft;
  const Plan pl = choose_plan(m > 0 ? m : 1, n > 0 ? n : 1, k > 0 ? k : 1, o->tile_n, want_sched,
                              want_grid, ms, 0, true, share, !o->abft && o->cta_pair != 2);
  r.sched = pl.sched;
  r.grid = pl.grid;
  r.grid_ck = 0;
  r.grid_ckt = 0;
  r.bn = pl.bn;
  r.pair = 0;
  r.grid_max = ms;
  r.share_min = kShareMin;
  r.share_bank2 = 0;
  // Split reduction for launches without ABFT; it takes the second region's
  // storage for owners' partials (bank 2), which compact workspaces leave out.
  r.split = (!o->abft && !compact) ? 1 : 0;
  r.ck_atomic = 0;
  if (o->cta_pair < 0 || o->cta_pair > 2) return SKG_ERR_ARG;
  if (o->cta_pair == 2 && o->tile_n != 0 && o->tile_n != 256) return SKG_ERR_UNSUPPORTED;
  bool use_pair = o->cta_pair == 2;
  if (o->cta_pair == 0 && o->grid == 0 && (o->tile_n == 0 || o->tile_n == 256) && sms > 0 &&
      m > 0 && n > 0 && k > 0) {
    // Automatic: pairs once their 256 x 256 tiles fill every resident
    // cluster at least once (measured faster from there; below, a wave of
    // 128-row tiles on more SMs wins).
    const int clusters = pair_clusters_resident();
    const int64_t ptiles = ((m + 2 * kBM - 1) / (2 * kBM)) * ((n + 255) / 256);
    use_pair = clusters > 0 && ptiles >= clusters;
  }
  if (use_pair) {
    // CTA pairs: the model plans 256-row tiles on the resident clusters.
    const int clusters = sms > 0 ? pair_clusters_resident() : ms / 2;
    if (clusters <= 0) return SKG_ERR_UNSUPPORTED;
    r.grid_max = 2 * clusters;
    if (o->grid > 0 && (o->grid % 2 != 0 || o->grid / 2 > clusters)) return SKG_ERR_UNSUPPORTED;
    const int want_pairs = o->grid > 0 ? o->grid / 2 : (want_sched >= 0 ? clusters : 0);
    const int64_t m_pairs = ((m > 0 ? m : 1) + 2 * kBM - 1) / (2 * kBM) * kBM;
    const Plan pp = choose_plan(m_pairs, n > 0 ? n : 1, k > 0 ? k : 1, 256, want_sched,
                                want_pairs, clusters, 0, true, share);
    r.pair = 1;
    r.bn = 256;
    r.sched = pp.sched;
    r.grid = 2 * pp.grid;
  }
  // With ABFT the checksum GEMMs may use every SM unless the caller fixes
  // the grid, which then bounds every launch of the call.
  r.ws_grid = (r.abft && o->grid == 0) ? (ms > r.grid ? ms : r.grid) : r.grid;
  r.k_for_plan = k > 0 ? k : 1;  // ABFT checksum GEMMs may use up to every SM
  r.tau_row = o->tau_row;
  r.tau_col = o->tau_col;
  const int32_t it[2] = {o->inject_tile, o->inject2_tile};
  const int32_t ir[2] = {o->inject_row, o->inject2_row};
  const int32_t ic[2] = {o->inject_col, o->inject2_col};
  const int32_t ib[2] = {o->inject_bit, o->inject2_bit};
  for (int sl = 0; sl < 2; ++sl) {
    r.inj_tile[sl] = it[sl] >= 0 ? it[sl] : -1;
    r.inj_row[sl] = ir[sl];
    r.inj_col[sl] = ic[sl];
    r.inj_bit[sl] = ib[sl];
    if (r.inj_tile[sl] >= 0 && (ir[sl] < 0 || ir[sl] >= kBM || ic[sl] < 0 || ic[sl] >= r.bn ||
                                ib[sl] < 0 || ib[sl] > 31))
      return SKG_ERR_ARG;
  }
  r.inj_kb = -1;
  if (o->inject_kstep >= 0 && r.inj_tile[0] >= 0) {
    if (o->inject_kstep >= (k + kBK - 1) / kBK) return SKG_ERR_ARG;
    r.inj_kb = o->inject_kstep;
  }
  if (o->stagger < 0) return SKG_ERR_ARG;
  r.stagger = o->stagger;
  r.timeout_ns = o->timeout_ns ? o->timeout_ns : kDefaultTimeoutNs;
  r.trace = o->trace;
  r.cta_clock = o->cta_clock;
  r.drop_signal = o->test_drop_signal - 1;
  r.preencoded = o->abft_preencoded ? 1 : 0;
  if (o->raster_band < 0) return SKG_ERR_ARG;
  r.raster_band = o->raster_band;
  r.enc_inkernel = 0;
  if (o->abft_local < 0 || o->abft_local > 2) return SKG_ERR_ARG;
  if (o->abft_inloop < 0 || o->abft_inloop > 2) return SKG_ERR_ARG;
  // In-loop reference checksums: a data-parallel plan over 128 x 128 tiles
  // on single CTAs or 256 x 256 tiles on CTA pairs (the choice above).
  r.ilc = 0;
  if (r.abft && o->abft_local != 2 && m > 0 && n > 0 && k > 0 &&
      (o->sched == SKG_SCHED_AUTO || o->sched == SKG_SCHED_DP) &&
      ilc_wanted(m, n, k, o, r, ms)) {
    if (r.pair) {
      const int clusters = r.grid_max / 2;
      const int64_t ptiles = ((m + 2 * kBM - 1) / (2 * kBM)) * ((n + 255) / 256);
      const int64_t want = o->grid > 0 ? o->grid / 2 : (ptiles < clusters ? ptiles : clusters);
      r.grid = 2 * (int)want;
      r.ilc = 1;
    } else if (o->tile_n == 0 || o->tile_n == 128) {
      const int64_t tiles = ((m + kBM - 1) / kBM) * ((n + 127) / 128);
      r.bn = 128;
      r.grid = o->grid > 0 ? o->grid : (int)(tiles < ms ? tiles : ms);
      r.ilc = 1;
    }
    if (r.ilc) {
      r.sched = SKG_SCHED_DP;
      r.grid_ck = 0;
      if (r.ws_grid < r.grid) r.ws_grid = r.grid;
    }
  }
  // In-CTA ABFT references (on request): a data-parallel plan of at most
  // one 128 x 128 tile per SM on single CTAs, so each CTA's epilogue warps
  // can read every stage of its one tile.
  r.abft_local = 0;
  if (r.abft && o->abft_local == 2 && m > 0 && n > 0 && k > 0 && o->cta_pair != 2 &&
      (o->tile_n == 0 || o->tile_n == 128) &&
      (o->sched == SKG_SCHED_AUTO || o->sched == SKG_SCHED_DP)) {
    const int64_t tiles = ((m + kBM - 1) / kBM) * ((n + 127) / 128);
    const bool fits = tiles <= ms && (o->grid == 0 || o->grid >= tiles);
    if (fits && r.inj_kb >= 0) return SKG_ERR_UNSUPPORTED;  // epilogue reads every stage
    if (fits) {
      r.abft_local = 1;
      r.bn = 128;
      r.sched = SKG_SCHED_DP;
      r.grid = (int)tiles;
      r.pair = 0;
      r.grid_max = ms;
      r.grid_ck = 0;
      const int bound = o->grid > 0 ? o->grid : ms;
      r.ws_grid = bound > r.grid ? bound : r.grid;
    }
  }
  return SKG_OK;
}

// Workspace layout. The header, the report and the flags (two regions of
// kMaxCtas) sit at fixed offsets for every shape and option set, so a
// workspace reused for another call finds only flags where its flags lie
// (their epochs keep them valid across launches). Everything after them is
// written by the call before the call reads it. Partial-tile slots are sized
// for the widest tile any launch of the call uses (the ABFT checksum GEMMs
// may use BLK_N = 256).
struct Layout {
  size_t flags, partials, sums, enc_a, enc_b, pub, umax, cr, cc, total;
  int kp, tiles_a, tiles_b;
  int64_t ld_cr, ld_cc;
};

constexpr size_t kFlagBytes = 2 * (size_t)kMaxCtas * 4;

Layout layout(int64_t m, int64_t n, int64_t k, const Resolved& r) {
  Layout L;
  size_t off = kHeaderBytes;
  // With ABFT the fused checksum tiles form a second split region with
  // flags and partial slots of its own.
  const size_t regions = (r.abft || r.share_bank2 || r.split) ? 2 : 1;
  L.flags = off;
  off += kFlagBytes;
  L.partials = off;
  const int slot_n = r.abft ? 256 : r.bn;
  off = round_up(off + regions * r.ws_grid * kBM * slot_n * 4, 256);
  L.kp = (int)round_up((size_t)(k > 0 ? k : 1), kBK);
  L.tiles_a = (int)((m + kBM - 1) / kBM);
  L.tiles_b = (int)((n + r.bn - 1) / r.bn);
  L.ld_cr = (int64_t)round_up((size_t)kEncRows * L.tiles_b, 4);
  L.ld_cc = (int64_t)round_up((size_t)kEncRows * L.tiles_a, 4);
  L.sums = L.enc_a = L.enc_b = L.pub = L.umax = L.cr = L.cc = off;
  if (r.abft) {
    const size_t tiles = (size_t)L.tiles_a + L.tiles_b;
    const size_t groups = (size_t)((m + kBM - 1) / kBM + (n + kBM - 1) / kBM);
    L.sums = off;
    off = round_up(off + groups * L.kp * 4, 256);
    L.enc_a = off;
    off = round_up(off + (size_t)kEncRows * L.tiles_a * L.kp * 2, 256);
    L.enc_b = off;
    off = round_up(off + (size_t)kEncRows * L.tiles_b * L.kp * 2, 256);
    L.pub = off;
    off = round_up(off + tiles * sizeof(TilePub), 256);
    L.umax = off;
    off = round_up(off + tiles * (size_t)encode_slices(L.kp) * 4, 256);
    L.cr = off;
    off = round_up(off + (size_t)m * L.ld_cr * 4, 256);
    L.cc = off;
    off = round_up(off + (size_t)n * L.ld_cc * 4, 256);
  }
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

CUresult make_map(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base,
                  uint64_t inner, uint64_t outer, uint64_t row_stride_elems, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_elems * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return tensor_map_encoder()(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// The ABFT encode pass over A (m x k) and the stored B (n x k).
skg_status_t run_encode(int32_t in_dtype, const void* A, int64_t lda, int64_t m, const void* B,
                        int64_t ldb, int64_t n, int64_t k, const Resolved& r, uint8_t* ws,
                        const Layout& L, int sms, cudaStream_t stream) {
  const CUtensorMapDataType in_t = in_dtype == SKG_IN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ma, mb;
  if (make_map(&ma, in_t, 2, A, (uint64_t)k, (uint64_t)m, (uint64_t)lda, kEncBoxCols, kEncBoxRows,
               CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
      make_map(&mb, in_t, 2, B, (uint64_t)k, (uint64_t)n, (uint64_t)ldb, kEncBoxCols, kEncBoxRows,
               CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return SKG_ERR_UNSUPPORTED;
  return launch_encode(in_dtype == SKG_IN_BF16, ma, mb, (int)m, (int)n, L.kp, r.bn, sms,
                       (float*)(ws + L.sums), ws + L.enc_a, ws + L.enc_b, (TilePub*)(ws + L.pub), (float*)(ws + L.umax), (skg_report_t*)(ws + 256),
                       r.timeout_ns,
                       stream) == cudaSuccess
             ? SKG_OK
             : SKG_ERR_CUDA;
}

// The encode pass for any operand layouts: one launch when both operands
// are K-major; otherwise each operand on its own, an MN-major one with the
// row-segment kernels and a K-major one with the pass above restricted to
// its tiles (the per-tile arrays offset past A's tiles for B).
skg_status_t run_encode_layouts(int32_t in_dtype, const void* A, int64_t lda, int a_mn, int64_t m,
                                const void* B, int64_t ldb, int b_mn, int64_t n, int64_t k,
                                const Resolved& r, uint8_t* ws, const Layout& L, int sms,
                                cudaStream_t stream) {
  if (!a_mn && !b_mn) return run_encode(in_dtype, A, lda, m, B, ldb, n, k, r, ws, L, sms, stream);
  const int bf16 = in_dtype == SKG_IN_BF16;
  const int slices = encode_slices(L.kp);
  float* sums = (float*)(ws + L.sums);
  float* umax = (float*)(ws + L.umax);
  TilePub* pub = (TilePub*)(ws + L.pub);
  const CUtensorMapDataType in_t = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cudaError_t e;
  if (a_mn) {
    e = launch_encode_mn(bf16, A, lda, m, k, kBM, L.tiles_a, L.kp, sums, umax, ws + L.enc_a, pub,
                         sms, stream);
  } else {
    CUtensorMap ma;
    if (make_map(&ma, in_t, 2, A, (uint64_t)k, (uint64_t)m, (uint64_t)lda, kEncBoxCols,
                 kEncBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return SKG_ERR_UNSUPPORTED;
    e = launch_encode(bf16, ma, ma, (int)m, 0, L.kp, r.bn, sms, sums, ws + L.enc_a, ws + L.enc_b,
                      pub, umax, (skg_report_t*)(ws + 256), r.timeout_ns, stream);
  }
  if (e != cudaSuccess) return SKG_ERR_CUDA;
  const int ta = L.tiles_a;
  if (b_mn) {
    e = launch_encode_mn(bf16, B, ldb, n, k, r.bn, L.tiles_b, L.kp, sums + (size_t)ta * L.kp,
                         umax + (size_t)ta * slices, ws + L.enc_b, pub + ta, sms, stream);
  } else {
    CUtensorMap mb;
    if (make_map(&mb, in_t, 2, B, (uint64_t)k, (uint64_t)n, (uint64_t)ldb, kEncBoxCols,
                 kEncBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return SKG_ERR_UNSUPPORTED;
    e = launch_encode(bf16, mb, mb, 0, (int)n, L.kp, r.bn, sms, sums + (size_t)ta * L.kp,
                      ws + L.enc_a, ws + L.enc_b, pub + ta,
                      umax + (size_t)ta * slices, (skg_report_t*)(ws + 256), r.timeout_ns,
                      stream);
  }
  return e == cudaSuccess ? SKG_OK : SKG_ERR_CUDA;
}

// One launch of the persistent kernel: C = alpha A B^T + beta C with A
// (m x k, row stride lda) and B (n x k, row stride ldb) in `in_dtype`.
struct Gemm {
  int64_t m, n, k;
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  void* C;
  int64_t ldc;
  float alpha, beta;
  int in_dtype, out_dtype;
  // MN-major operands read directly by the MMAs (A stored k x m, B stored
  // k x n), in the output tiles and as the A operand of the checksum tiles.
  int a_mn = 0, b_mn = 0;
};

template <int BN, bool ABFT, bool PAIR = false, bool LOCAL = false, bool MN = false,
          bool ILC = false>
cudaError_t dispatch_out(int out_dtype, const Maps& mp, const KernelParams& p, int grid,
                         cudaStream_t st) {
  switch (out_dtype) {
    case SKG_OUT_F32: return launch_gemm<BN, ABFT, 0, PAIR, LOCAL, MN, ILC>(mp, p, grid, st);
    case SKG_OUT_F16: return launch_gemm<BN, ABFT, 1, PAIR, LOCAL, MN, ILC>(mp, p, grid, st);
    default: return launch_gemm<BN, ABFT, 2, PAIR, LOCAL, MN, ILC>(mp, p, grid, st);
  }
}

// The instantiation for the launch's operand layouts: K-major kernels carry
// no MN-major code.
template <int BN, bool ABFT, bool PAIR = false>
cudaError_t dispatch_layout(bool mn, int out_dtype, const Maps& mp, const KernelParams& p,
                            int grid, cudaStream_t st) {
  return mn ? dispatch_out<BN, ABFT, PAIR, false, true>(out_dtype, mp, p, grid, st)
            : dispatch_out<BN, ABFT, PAIR>(out_dtype, mp, p, grid, st);
}

// Fused ABFT checksum GEMMs fit one tile column each when 2 * tiles <= BN.
bool can_fuse_checksums(const Layout& L, int bn) {
  return kEncRows * L.tiles_a <= bn && kEncRows * L.tiles_b <= bn;
}

// One launch of the persistent kernel: C = alpha A B^T + beta C with A
// (m x k, row stride lda) and B (n x k, row stride ldb) in `in_dtype`.
// With fuse_ck, the tiles of the two ABFT checksum GEMMs are scheduled in
// front of the output tiles of the same launch.
skg_status_t launch_one(const Gemm& g, const Resolved& r, bool abft_epilogue, bool fuse_ck,
                        uint8_t* ws, const Layout& L, cudaStream_t stream) {
  const CUtensorMapDataType in_t = g.in_dtype == SKG_IN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType out_t = g.out_dtype == SKG_OUT_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : g.out_dtype == SKG_OUT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int out_bytes = g.out_dtype == SKG_OUT_F32 ? 4 : 2;
  Maps mp;
  // K-major operands: one kBK x rows box per stage; MN-major ones: boxes of
  // 64 MN elements x kBK (the kernel issues rows / 64 of them).
  const CUresult ra =
      g.a_mn ? make_map(&mp.a, in_t, 2, g.A, (uint64_t)g.m, (uint64_t)g.k, (uint64_t)g.lda,
                        kMnBox, kBK)
             : make_map(&mp.a, in_t, 2, g.A, (uint64_t)g.k, (uint64_t)g.m, (uint64_t)g.lda, kBK,
                        kBM);
  const CUresult rb =
      g.b_mn ? make_map(&mp.b, in_t, 2, g.B, (uint64_t)g.n, (uint64_t)g.k, (uint64_t)g.ldb,
                        kMnBox, kBK)
             : make_map(&mp.b, in_t, 2, g.B, (uint64_t)g.k, (uint64_t)g.n, (uint64_t)g.ldb, kBK,
                        r.pair ? r.bn / 2 : r.bn);
  if (ra != CUDA_SUCCESS || rb != CUDA_SUCCESS ||
      make_map(&mp.c, out_t, out_bytes, g.C, (uint64_t)g.n, (uint64_t)g.m, (uint64_t)g.ldc,
               128 / out_bytes, 32) != CUDA_SUCCESS)
    return SKG_ERR_UNSUPPORTED;
  mp.b128 = mp.be = mp.ea = mp.cr = mp.cc = mp.enca = mp.encb = mp.a;
  int t_ck = 0, ck_cr = 0;
  // CTA pairs: a side tile is two 128-row checksum tiles, the encoding rows
  // (the MMA's N) are split between the two CTAs, so N rounds up to 32.
  const int ck_half = r.pair ? 2 : 1;
  const int ck_round = r.pair ? 32 : 16;
  if (fuse_ck) {
    const int n_cr = kEncRows * L.tiles_b, n_cc = kEncRows * L.tiles_a;
    const CUresult rb128 =
        g.b_mn ? make_map(&mp.b128, in_t, 2, g.B, (uint64_t)g.n, (uint64_t)g.k,
                          (uint64_t)g.ldb, kMnBox, kBK)
               : make_map(&mp.b128, in_t, 2, g.B, (uint64_t)g.k, (uint64_t)g.n,
                          (uint64_t)g.ldb, kBK, kBM);
    if (rb128 != CUDA_SUCCESS ||
        make_map(&mp.be, in_t, 2, ws + L.enc_b, (uint64_t)L.kp, (uint64_t)n_cr, (uint64_t)L.kp,
                 kBK, (uint32_t)(round_up(n_cr, ck_round) / ck_half)) != CUDA_SUCCESS ||
        make_map(&mp.ea, in_t, 2, ws + L.enc_a, (uint64_t)L.kp, (uint64_t)n_cc, (uint64_t)L.kp,
                 kBK, (uint32_t)(round_up(n_cc, ck_round) / ck_half)) != CUDA_SUCCESS ||
        make_map(&mp.cr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws + L.cr, (uint64_t)n_cr,
                 (uint64_t)g.m, (uint64_t)L.ld_cr, 32, 32) != CUDA_SUCCESS ||
        make_map(&mp.cc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws + L.cc, (uint64_t)n_cc,
                 (uint64_t)g.n, (uint64_t)L.ld_cc, 32, 32) != CUDA_SUCCESS)
      return SKG_ERR_UNSUPPORTED;
    ck_cr = (int)(((g.m + kBM - 1) / kBM + ck_half - 1) / ck_half);
    t_ck = ck_cr + (int)(((g.n + kBM - 1) / kBM + ck_half - 1) / ck_half);
  }

  // In-loop checksums: the encodings of one k-step (hi and lo rows) are
  // loaded with each stage as the N = 16 operand of the checksum MMAs.
  const bool ilc = abft_epilogue && r.ilc;
  if (ilc &&
      (make_map(&mp.ea, in_t, 2, ws + L.enc_a, (uint64_t)L.kp, (uint64_t)kEncRows * L.tiles_a,
                (uint64_t)L.kp, kBK, kEncRows) != CUDA_SUCCESS ||
       make_map(&mp.be, in_t, 2, ws + L.enc_b, (uint64_t)L.kp, (uint64_t)kEncRows * L.tiles_b,
                (uint64_t)L.kp, kBK, kEncRows) != CUDA_SUCCESS))
    return SKG_ERR_UNSUPPORTED;

  KernelParams p;
  memset(&p, 0, sizeof(p));
  // CTA pairs: 256-row tiles, one schedule CTA per cluster.
  const int sched_ctas = r.pair ? r.grid / 2 : r.grid;
  p.s = make_schedule(g.m, g.n, g.k, r.pair ? 2 * kBM : kBM, r.bn, kBK, sched_ctas, r.sched, t_ck,
                      t_ck ? r.grid_ck : 0, t_ck ? r.grid_ckt : -1);
  const int launch_grid = r.grid + p.s.g_ck;
  if (launch_grid > kMaxCtas) return SKG_ERR_UNSUPPORTED;  // flags per region
  // Banded raster: a wave of g tiles covers about (g / band) rows x band
  // columns; band ~ sqrt(g * BLK_M / BLK_N) minimises the A + B bytes one
  // wave touches per k-step.
  int band = r.raster_band;
  if (band == 0) {
    const double b = sqrt((double)sched_ctas * (r.pair ? 2 * kBM : kBM) / r.bn);
    band = (int)(b + 0.5);
  }
  if (band < 1) band = 1;
  if (band < p.s.tiles_n) p.s.band = band;
  if (!abft_epilogue) {
    p.s.share_min = r.share_min;
    p.s.share_bank2 = (r.share_bank2 || r.split) ? 1 : 0;
    // Split parts own whole staging chunks (BLK_N / EPI_COLS of them).
    p.s.split_max = (r.split && !r.pair) ? r.bn * out_bytes / 128 : 0;
  }
  p.m = (int)g.m;
  p.n = (int)g.n;
  p.k = (int)g.k;
  p.alpha = g.alpha;
  p.beta = g.beta;
  p.idesc_main = idesc_f16(g.in_dtype == SKG_IN_BF16, r.pair ? 2 * kBM : kBM, r.bn) |
                 ((uint32_t)(g.a_mn != 0) << 15) | ((uint32_t)(g.b_mn != 0) << 16);
  p.a_mn = g.a_mn;
  p.b_mn = g.b_mn;
  p.ck_cr_tiles = ck_cr;
  p.ck_n_cr = kEncRows * L.tiles_b;
  p.ck_n_cc = kEncRows * L.tiles_a;
  p.ck_rows_cr = (int)round_up(p.ck_n_cr, ck_round);
  p.ck_rows_cc = (int)round_up(p.ck_n_cc, ck_round);
  // Two checksum k-blocks per ring stage when the encoding box fits its
  // 8 KB slot (64 rows of 128 bytes) and the stage holds two A tiles.
  p.ck_kpack_cr = (!r.pair && r.bn == 256 && p.ck_rows_cr <= 64) ? 2 : 1;
  p.ck_kpack_cc = (!r.pair && r.bn == 256 && p.ck_rows_cc <= 64) ? 2 : 1;
  p.ck_atomic = (fuse_ck && r.ck_atomic && r.enc_inkernel) ? 1 : 0;
  if (p.ck_atomic) {
    // Segment reports the verifying epilogues wait for: one per (CTA,
    // checksum tile) piece of the side region's split.
    const Schedule& cs = p.s;
    const int split_ctas = (cs.g_ck > 0 && cs.g_ckt > 0) ? cs.g_ckt : cs.g;
    int64_t segs = 0;
    for (int x = 0; x < split_ctas; ++x) {
      int64_t b, e;
      even_range(cs.ck_q, cs.ck_r, x, b, e);
      if (e > b) segs += (e - 1) / cs.ipt - b / cs.ipt + 1;
    }
    p.ck_target = (int)(segs * ck_half);
  }
  // The checksum tiles' A operand is A (cr) or B (cc), MN-major as stored.
  p.idesc_cr = idesc_f16(g.in_dtype == SKG_IN_BF16, ck_half * kBM, (uint32_t)p.ck_rows_cr) |
               ((uint32_t)(g.a_mn != 0) << 15);
  p.idesc_cc = idesc_f16(g.in_dtype == SKG_IN_BF16, ck_half * kBM, (uint32_t)p.ck_rows_cc) |
               ((uint32_t)(g.b_mn != 0) << 15);
  if (ilc) {  // checksum MMAs of the output tiles: M = the tile's rows, N = 16
    p.idesc_cr = idesc_f16(g.in_dtype == SKG_IN_BF16, r.pair ? 2 * kBM : kBM, 16);
    p.idesc_cc = p.idesc_cr;
  }
  p.hdr = (WsHeader*)ws;
  p.report = (skg_report_t*)(ws + 256);
  p.flags = (uint32_t*)(ws + L.flags);
  p.partials = (float*)(ws + L.partials);
  p.ws_ctas = r.ws_grid;
  p.cr_all = (const float*)(ws + L.cr);
  p.cc_all = (const float*)(ws + L.cc);
  p.ld_cr = L.ld_cr;
  p.ld_cc = L.ld_cc;
  p.pub_a = (const TilePub*)(ws + L.pub);
  p.pub_b = (const TilePub*)(ws + L.pub) + L.tiles_a;
  p.umax = (const float*)(ws + L.umax);
  p.enc_slices = encode_slices(L.kp);
  p.enc_tiles_a = L.tiles_a;
  if (fuse_ck && r.enc_inkernel) {
    if (make_map(&mp.enca, in_t, 2, g.A, (uint64_t)g.k, (uint64_t)g.m, (uint64_t)g.lda,
                 kEncBoxCols, kEncBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
        make_map(&mp.encb, in_t, 2, g.B, (uint64_t)g.k, (uint64_t)g.n, (uint64_t)g.ldb,
                 kEncBoxCols, kEncBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return SKG_ERR_UNSUPPORTED;
    p.enc_inkernel = 1;
    p.enc_tiles_b = L.tiles_b;
    p.enc_bn = r.bn;
    p.enc_kp = L.kp;
    p.enc_a_w = ws + L.enc_a;
    p.enc_b_w = ws + L.enc_b;
    p.umax_w = (float*)(ws + L.umax);
    p.pub_w = (TilePub*)(ws + L.pub);
  }
  p.tau_row = r.tau_row;
  p.tau_col = r.tau_col;
  for (int sl = 0; sl < 2; ++sl) {
    p.inj_tile[sl] = r.inj_tile[sl];
    p.inj_row[sl] = r.inj_row[sl];
    p.inj_col[sl] = r.inj_col[sl];
    p.inj_bit[sl] = r.inj_bit[sl];
  }
  p.inj_kb = r.inj_kb;
  p.stagger = r.stagger;
  p.timeout_ns = r.timeout_ns;
  p.trace = r.trace;
  p.cta_clock = r.cta_clock;
  p.drop_signal = r.drop_signal;
  p.c_ptr = g.C;
  p.ldc = g.ldc;
  p.in_f16 = g.in_dtype == SKG_IN_F16 ? 1 : 0;

  const bool mn = g.a_mn || g.b_mn;
  const int od = g.out_dtype;
  const int lg = launch_grid;
  cudaError_t e;
  if (ilc)
    e = r.pair ? dispatch_out<256, true, true, false, false, true>(od, mp, p, lg, stream)
               : dispatch_out<128, true, false, false, false, true>(od, mp, p, lg, stream);
  else if (r.pair)
    e = abft_epilogue ? dispatch_layout<256, true, true>(mn, od, mp, p, lg, stream)
                      : dispatch_layout<256, false, true>(mn, od, mp, p, lg, stream);
  else if (r.bn == 64)
    e = abft_epilogue ? cudaErrorInvalidValue  // resolve() keeps ABFT off 64-wide tiles
                      : dispatch_layout<64, false>(mn, od, mp, p, lg, stream);
  else if (r.bn == 128)
    e = (abft_epilogue && r.abft_local && !fuse_ck)
            ? dispatch_out<128, true, false, true>(od, mp, p, lg, stream)
        : abft_epilogue ? dispatch_layout<128, true>(mn, od, mp, p, lg, stream)
                        : dispatch_layout<128, false>(mn, od, mp, p, lg, stream);
  else
    e = abft_epilogue ? dispatch_layout<256, true>(mn, od, mp, p, lg, stream)
                      : dispatch_layout<256, false>(mn, od, mp, p, lg, stream);
  return e == cudaSuccess ? SKG_OK : SKG_ERR_CUDA;
}

// The ABFT reference checksums of every output tile ("Anatomy of
// High-Performance GEMM with Online Fault Tolerance on GPUs", Fig. 3:
// C^r = A (B e), C^c = (e^T A) B): the encode pass, then two tall-skinny
// GEMMs on the same persistent kernel with fp32 output, each reading its
// large operand once:
//   cr_all  (m x 2 tiles_b) = A x [Be_hi; Be_lo]^T
//   ccT_all (n x 2 tiles_a) = B x [eA_hi; eA_lo]^T     (= ((e^T A) B)^T)
skg_status_t reference_checksums(const Gemm& g, const Resolved& r, uint8_t* ws, const Layout& L,
                                 cudaStream_t stream, bool skip_encode) {
  if (!skip_encode) {
    const skg_status_t st =
        run_encode_layouts(g.in_dtype, g.A, g.lda, g.a_mn, g.m, g.B, g.ldb, g.b_mn, g.n, g.k, r,
                           ws, L, sm_count_cached(), stream);
    if (st != SKG_OK) return st;
  }
  Resolved rc = r;
  rc.abft = 0;
  rc.pair = 0;
  rc.inj_tile[0] = rc.inj_tile[1] = -1;
  rc.inj_kb = -1;
  rc.stagger = 0;
  rc.trace = nullptr;
  rc.cta_clock = nullptr;
  rc.drop_signal = -1;
  rc.raster_band = 0;
  Gemm g1{g.m, (int64_t)kEncRows * L.tiles_b, g.k, g.A, g.lda, ws + L.enc_b, L.kp,
          ws + L.cr, L.ld_cr, 1.f, 0.f, g.in_dtype, SKG_OUT_F32};
  g1.a_mn = g.a_mn;  // the encodings (B operand) are K-major
  Plan pl = choose_plan(g1.m, g1.n, g1.k, 0, -1, 0, r.ws_grid);
  rc.bn = pl.bn;
  rc.sched = pl.sched;
  rc.grid = pl.grid;
  skg_status_t st = launch_one(g1, rc, false, false, ws, L, stream);
  if (st != SKG_OK) return st;
  Gemm g2{g.n, (int64_t)kEncRows * L.tiles_a, g.k, g.B, g.ldb, ws + L.enc_a, L.kp,
          ws + L.cc, L.ld_cc, 1.f, 0.f, g.in_dtype, SKG_OUT_F32};
  g2.a_mn = g.b_mn;  // B as the A operand
  pl = choose_plan(g2.m, g2.n, g2.k, 0, -1, 0, r.ws_grid);
  rc.bn = pl.bn;
  rc.sched = pl.sched;
  rc.grid = pl.grid;
  return launch_one(g2, rc, false, false, ws, L, stream);
}

// With fused checksum tiles the launch has tiles_a + ceil(n / 128) more
// full-k tiles; re-plan the grid (and schedule) for them unless fixed.
void replan_fused(int64_t m, int64_t n, const skg_opts_t* opts, Resolved& r) {
  skg_opts_t d;
  if (!opts) {
    skg_opts_default(&d);
    opts = &d;
  }
  if (opts->grid != 0) return;
  const int want_sched = opts->sched == SKG_SCHED_AUTO ? -1 : opts->sched;
  if (r.pair) {
    // 256-row tiles and pair side tiles on the resident clusters; the side
    // tiles are always split over the grid (no dedicated CTAs).
    const int clusters = r.grid_max / 2;
    const int64_t tm = (m + kBM - 1) / kBM, tn = (n + kBM - 1) / kBM;
    const int t_ck = (int)((tm + 1) / 2 + (tn + 1) / 2);
    const int64_t m_pairs = (m + 2 * kBM - 1) / (2 * kBM) * kBM;
    const Plan pp = choose_plan(m_pairs, n, r.k_for_plan, 256, want_sched,
                                want_sched >= 0 ? clusters : 0, clusters, t_ck, false, false);
    r.grid = 2 * pp.grid;
    r.sched = pp.sched;
    r.grid_ck = 0;
    return;
  }
  const int t_ck = (int)((m + kBM - 1) / kBM + (n + kBM - 1) / kBM);
  const Plan pl = choose_plan(m, n, r.k_for_plan, r.bn, want_sched,
                              want_sched >= 0 ? r.ws_grid : 0, r.ws_grid, t_ck, true, false);
  r.grid = pl.grid;
  r.sched = pl.sched;
  r.grid_ck = pl.grid_ck;
  r.grid_ckt = pl.grid_ck;
}

// Plan of a call whose checksum GEMMs are fused: grid and schedule with the
// side tiles, then their placement. Checksum tiles on dedicated CTAs leave
// SMs idle while the output tiles run, so those CTAs take every idle SM and
// the encode pass too (bf16 encodings need no per-tile scale).
void plan_fused(int64_t m, int64_t n, const skg_opts_t* opts, int32_t in_dtype, bool k_major,
                Resolved& r) {
  replan_fused(m, n, opts, r);
  // Only with plenty of idle SMs (at least four per checksum tile): the
  // side CTAs' encode-then-checksum chain must end with the output tiles.
  r.enc_inkernel = (k_major && !r.preencoded && r.grid_ck > 0 && !r.pair &&
                    in_dtype == SKG_IN_BF16 &&
                    r.grid_max - r.grid >= 4 * r.grid_ck && kEncBoxCols == kEncInCols &&
                    kEncBoxRows == kEncInRows)
                       ? 1
                       : 0;
  if (r.enc_inkernel) r.grid_ck = r.grid_max - r.grid;
  // With the encode pass in this launch its CTAs also zero the reference
  // arrays, so the checksum tiles can be split over all of the side CTAs
  // with each segment adding its rows in (no owner waits for its peers):
  // measured 2 us shorter at 1024^3 than whole checksum tiles on t_ck CTAs.
  if (r.enc_inkernel) {
    r.ck_atomic = 1;
    r.grid_ckt = r.grid_ck;
  }
}

// Whether an ABFT call runs on K-major copies of its MN-major operands.
// Everything else reads them in place; two paths read K-major stages only:
// the in-CTA references (epilogue warps read the stages as K-major rows) and
// the in-kernel encode pass of dedicated side CTAs. Where the plan would use
// the latter (small bf16 shapes with many idle SMs), two short copies and
// one launch beat the separate MN-major encode launches.
bool abft_wants_copies(int64_t m, int64_t n, const skg_opts_t* opts, int32_t in_dtype,
                       const Resolved& r, const Layout& L) {
  if (!r.abft) return false;
  if (r.abft_local) return true;
  if (!can_fuse_checksums(L, r.bn)) return false;
  Resolved probe = r;
  plan_fused(m, n, opts, in_dtype, true, probe);
  return probe.enc_inkernel != 0;
}

skg_status_t check_inputs(int64_t m, int64_t n, int64_t k, const void* A, int64_t lda,
                          const void* B, int64_t ldb, int32_t a_layout = SKG_A_ROW,
                          int32_t b_layout = SKG_B_KMAJOR) {
  if (!A || !B) return SKG_ERR_ARG;
  // The leading dimension spans the operand's contiguous index: k for the
  // K-major forms, m (A column-major) or n (B stored k x n) otherwise.
  if (lda < (a_layout == SKG_A_COL ? m : k) || ldb < (b_layout == SKG_B_NMAJOR ? n : k))
    return SKG_ERR_ARG;
  if (!aligned16(A) || !aligned16(B) || (lda * 2) % 16 || (ldb * 2) % 16)
    return SKG_ERR_UNSUPPORTED;
  return SKG_OK;
}

// K-major copies of MN-major operands, placed after the rest of the
// workspace: A as m x ldk, B as n x ldk (ldk = k rounded up to 8 elements,
// so rows start on 16-byte boundaries as the TMA engine requires).
struct Relayout {
  size_t a = 0, b = 0, total = 0;  // offsets from the workspace base; total = end
  int64_t ldk = 0;
};

Relayout relayout_plan(int64_t m, int64_t n, int64_t k, int32_t a_layout, int32_t b_layout,
                       size_t base) {
  Relayout R;
  R.ldk = (int64_t)round_up((size_t)(k > 0 ? k : 1), 8);
  size_t off = round_up(base, 256);
  if (a_layout == SKG_A_COL) {
    R.a = off;
    off = round_up(off + (size_t)m * R.ldk * 2, 256);
  }
  if (b_layout == SKG_B_NMAJOR) {
    R.b = off;
    off = round_up(off + (size_t)n * R.ldk * 2, 256);
  }
  R.total = (a_layout == SKG_A_COL || b_layout == SKG_B_NMAJOR) ? off : base;
  return R;
}

// The layout whose operand gets a K-major copy (`copies`, below): the
// MN-major ones, or none.
int32_t copy_layout_a(int32_t a_layout, bool copies) { return copies ? a_layout : SKG_A_ROW; }
int32_t copy_layout_b(int32_t b_layout, bool copies) {
  return copies ? b_layout : SKG_B_KMAJOR;
}

bool layout_valid(int32_t a_layout, int32_t b_layout) {
  return (a_layout == SKG_A_ROW || a_layout == SKG_A_COL) &&
         (b_layout == SKG_B_KMAJOR || b_layout == SKG_B_NMAJOR);
}

// Device staging of skg_gemm_host: packed copies of A and B as stored and
// of C, each row rounded up to 16 bytes.
struct Staging {
  int64_t a_rows, a_cols, b_rows, b_cols;  // stored shapes (elements)
  int64_t lda, ldb, ldc;                   // device leading dimensions
  size_t a, b, c, total;                   // byte offsets, total size
  int out_bytes;
};

bool staging_plan(int64_t m, int64_t n, int64_t k, int32_t in_dtype, int32_t out_dtype,
                  int32_t a_layout, int32_t b_layout, Staging& S) {
  if (m < 0 || n < 0 || k < 0) return false;
  if (in_dtype != SKG_IN_F16 && in_dtype != SKG_IN_BF16) return false;
  if (out_dtype < SKG_OUT_F32 || out_dtype > SKG_OUT_BF16) return false;
  if (!layout_valid(a_layout, b_layout)) return false;
  S.out_bytes = out_dtype == SKG_OUT_F32 ? 4 : 2;
  S.a_rows = a_layout == SKG_A_ROW ? m : k;
  S.a_cols = a_layout == SKG_A_ROW ? k : m;
  S.b_rows = b_layout == SKG_B_KMAJOR ? n : k;
  S.b_cols = b_layout == SKG_B_KMAJOR ? k : n;
  S.lda = (int64_t)round_up((size_t)(S.a_cols > 0 ? S.a_cols : 1), 8);
  S.ldb = (int64_t)round_up((size_t)(S.b_cols > 0 ? S.b_cols : 1), 8);
  S.ldc = (int64_t)round_up((size_t)(n > 0 ? n : 1), (size_t)(16 / S.out_bytes));
  size_t off = 0;
  S.a = off;
  off = round_up(off + (size_t)S.a_rows * S.lda * 2, 256);
  S.b = off;
  off = round_up(off + (size_t)S.b_rows * S.ldb * 2, 256);
  S.c = off;
  off = round_up(off + (size_t)m * S.ldc * S.out_bytes, 256);
  S.total = off;
  return true;
}

skg_status_t gemm_impl(int64_t m, int64_t n, int64_t k, float alpha, const void* A, int64_t lda,
                       const void* B, int64_t ldb, float beta, void* C, int64_t ldc,
                       int32_t in_dtype, int32_t out_dtype, int32_t a_layout, int32_t b_layout,
                       const skg_opts_t* opts, int force_abft, void* workspace,
                       size_t ws_bytes, void* stream_v, bool compact = false) {
  cudaStream_t stream = (cudaStream_t)stream_v;
  if (m < 0 || n < 0 || k < 0) return SKG_ERR_ARG;
  if (m > INT32_MAX / 4 || n > INT32_MAX / 4 || k > INT32_MAX / 4) return SKG_ERR_UNSUPPORTED;
  if (in_dtype != SKG_IN_F16 && in_dtype != SKG_IN_BF16) return SKG_ERR_ARG;
  if (out_dtype < SKG_OUT_F32 || out_dtype > SKG_OUT_BF16) return SKG_ERR_ARG;
  if (!layout_valid(a_layout, b_layout)) return SKG_ERR_ARG;
  if (m == 0 || n == 0) return SKG_OK;
  const int out_bytes = out_dtype == SKG_OUT_F32 ? 4 : 2;
  if (!C) return SKG_ERR_ARG;
  if (ldc < n) return SKG_ERR_ARG;
  if (!aligned16(C) || (ldc * out_bytes) % 16) return SKG_ERR_UNSUPPORTED;
  if (k == 0) {
    return launch_scale(out_dtype, C, ldc, (int)m, (int)n, beta, stream) == cudaSuccess
               ? SKG_OK
               : SKG_ERR_CUDA;
  }
  skg_status_t st = check_inputs(m, n, k, A, lda, B, ldb, a_layout, b_layout);
  if (st != SKG_OK) return st;

  const int sms = sm_count_cached();
  if (sms <= 0) return SKG_ERR_CUDA;
  Resolved r;
  skg_opts_t forced;
  if (force_abft) {
    if (opts) forced = *opts;
    else skg_opts_default(&forced);
    forced.abft = 1;
    opts = &forced;
  }
  st = resolve(m, n, k, opts, r, sms, compact);
  if (st != SKG_OK) return st;
  const Layout L = layout(m, n, k, r);
  const bool copies = (a_layout == SKG_A_COL || b_layout == SKG_B_NMAJOR) &&
                      abft_wants_copies(m, n, opts, in_dtype, r, L);
  const Relayout R = relayout_plan(m, n, k, copy_layout_a(a_layout, copies),
                                   copy_layout_b(b_layout, copies), L.total);
  if (!workspace || !aligned16(workspace) || ws_bytes < R.total) return SKG_ERR_WORKSPACE;
  if (!tensor_map_encoder()) return SKG_ERR_CUDA;

  uint8_t* ws = (uint8_t*)workspace;
  // MN-major operands are read in place (output and checksum tiles, encode
  // pass) unless abft_wants_copies: then the call runs on K-major copies in
  // the workspace.
  if (copy_layout_a(a_layout, copies) == SKG_A_COL) {
    if (launch_relayout(A, lda, m, k, ws + R.a, R.ldk, sms, stream) != cudaSuccess)
      return SKG_ERR_CUDA;
    A = ws + R.a;
    lda = R.ldk;
  }
  if (copy_layout_b(b_layout, copies) == SKG_B_NMAJOR) {
    if (launch_relayout(B, ldb, n, k, ws + R.b, R.ldk, sms, stream) != cudaSuccess)
      return SKG_ERR_CUDA;
    B = ws + R.b;
    ldb = R.ldk;
  }
  Gemm g{m, n, k, A, lda, B, ldb, C, ldc, alpha, beta, in_dtype, out_dtype};
  g.a_mn = !copies && a_layout == SKG_A_COL;
  g.b_mn = !copies && b_layout == SKG_B_NMAJOR;
  bool fuse = false;
  if (r.ilc && (g.a_mn || g.b_mn)) r.ilc = 0;  // in-loop checksums read K-major stages
  if (r.abft && r.abft_local) {
    // The reference checksums are formed inside the CTAs: one launch.
  } else if (r.abft && r.ilc) {
    // The encode pass, then one launch whose MMAs also accumulate the
    // reference checksums.
    if (!r.preencoded) {
      st = run_encode_layouts(in_dtype, A, lda, 0, m, B, ldb, 0, n, k, r, ws, L, sms, stream);
      if (st != SKG_OK) return st;
    }
  } else if (r.abft && can_fuse_checksums(L, r.bn)) {
    // The checksum-GEMM tiles run ahead of the output tiles in the same
    // launch, after the encode pass (skipped when pre-encoded).
    fuse = true;
    plan_fused(m, n, opts, in_dtype, !g.a_mn && !g.b_mn, r);
    if (!r.enc_inkernel && !r.preencoded) {
      st = run_encode_layouts(in_dtype, A, lda, g.a_mn, m, B, ldb, g.b_mn, n, k, r, ws, L, sms,
                              stream);
      if (st != SKG_OK) return st;
    }
  } else if (r.abft) {
    st = reference_checksums(g, r, ws, L, stream, r.preencoded != 0);
    if (st != SKG_OK) return st;
  }
  return launch_one(g, r, r.abft != 0, fuse, ws, L, stream);
}

}  // namespace

namespace skg {

skg_status_t workspace_need(int64_t m, int64_t n, int64_t k, int32_t a_layout, int32_t b_layout,
                            const skg_opts_t* opts, size_t* need, bool compact) {
  if (!layout_valid(a_layout, b_layout)) return SKG_ERR_ARG;
  if (m < 0 || n < 0 || k < 0) return SKG_ERR_ARG;
  Resolved r;
  const int sms = sm_count_cached();
  const skg_status_t st = resolve(m, n, k, opts, r, sms, compact);
  if (st != SKG_OK) return st;
  const Layout L = layout(m, n, k, r);
  // The copies are planned for bf16, the input type for which they can be
  // chosen (abft_wants_copies), so the size covers either type.
  const bool copies = (a_layout == SKG_A_COL || b_layout == SKG_B_NMAJOR) &&
                      abft_wants_copies(m, n, opts, SKG_IN_BF16, r, L);
  *need = relayout_plan(m, n, k, copy_layout_a(a_layout, copies),
                        copy_layout_b(b_layout, copies), L.total)
              .total;
  return SKG_OK;
}

size_t fixed_header_bytes() { return kHeaderBytes + kFlagBytes; }

skg_status_t gemm_compact(int64_t m, int64_t n, int64_t k, float alpha, const void* A,
                          int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                          int64_t ldc, int32_t in_dtype, int32_t out_dtype, int32_t a_layout,
                          int32_t b_layout, const skg_opts_t* opts, void* workspace,
                          size_t ws_bytes, void* stream) {
  return gemm_impl(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, a_layout,
                   b_layout, opts, 0, workspace, ws_bytes, stream, true);
}

}  // namespace skg

extern "C" {

void skg_opts_default(skg_opts_t* o) {
  if (!o) return;
  memset(o, 0, sizeof(*o));
  o->sched = SKG_SCHED_AUTO;
  o->inject_tile = -1;
  o->inject2_tile = -1;
  o->inject_kstep = -1;
}

size_t skg_workspace_size(int64_t m, int64_t n, int64_t k, const skg_opts_t* opts) {
  if (m < 0 || n < 0 || k < 0) return 0;
  Resolved r;
  const int sms = sm_count_cached();
  if (resolve(m, n, k, opts, r, sms) != SKG_OK) return 0;
  return layout(m, n, k, r).total;
}

size_t skg_workspace_size_layout(int64_t m, int64_t n, int64_t k, int32_t a_layout,
                                 int32_t b_layout, const skg_opts_t* opts) {
  size_t need = 0;
  return skg::workspace_need(m, n, k, a_layout, b_layout, opts, &need) == SKG_OK ? need : 0;
}

skg_status_t skg_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace || bytes < kHeaderBytes) return SKG_ERR_WORKSPACE;
  return cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream) == cudaSuccess ? SKG_OK
                                                                                 : SKG_ERR_CUDA;
}

skg_status_t skg_gemm(int64_t m, int64_t n, int64_t k, float alpha, const void* A, int64_t lda,
                      const void* B, int64_t ldb, float beta, void* C, int64_t ldc,
                      int32_t in_dtype, int32_t out_dtype, int32_t a_layout, int32_t b_layout,
                      const skg_opts_t* opts, void* workspace, size_t ws_bytes, void* stream) {
  return gemm_impl(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, a_layout,
                   b_layout, opts, 0, workspace, ws_bytes, stream);
}

skg_status_t skg_gemm_verify(int64_t m, int64_t n, int64_t k, float alpha, const void* A,
                             int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                             int64_t ldc, int32_t in_dtype, int32_t out_dtype, int32_t a_layout,
                             int32_t b_layout, const skg_opts_t* opts, void* workspace,
                             size_t ws_bytes, void* stream) {
  return gemm_impl(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, in_dtype, out_dtype, a_layout,
                   b_layout, opts, 1, workspace, ws_bytes, stream);
}

skg_status_t skg_abft_encode(int64_t m, int64_t n, int64_t k, const void* A, int64_t lda,
                             const void* B, int64_t ldb, int32_t in_dtype,
                             const skg_opts_t* opts, void* workspace, size_t ws_bytes,
                             void* stream) {
  return skg_abft_encode_layout(m, n, k, A, lda, B, ldb, in_dtype, SKG_A_ROW, SKG_B_KMAJOR, opts,
                                workspace, ws_bytes, stream);
}

skg_status_t skg_abft_encode_layout(int64_t m, int64_t n, int64_t k, const void* A, int64_t lda,
                                    const void* B, int64_t ldb, int32_t in_dtype,
                                    int32_t a_layout, int32_t b_layout, const skg_opts_t* opts,
                                    void* workspace, size_t ws_bytes, void* stream) {
  if (m < 0 || n < 0 || k < 0) return SKG_ERR_ARG;
  if (m > INT32_MAX / 4 || n > INT32_MAX / 4 || k > INT32_MAX / 4) return SKG_ERR_UNSUPPORTED;
  if (in_dtype != SKG_IN_F16 && in_dtype != SKG_IN_BF16) return SKG_ERR_ARG;
  if (!layout_valid(a_layout, b_layout)) return SKG_ERR_ARG;
  if (m == 0 || n == 0 || k == 0) return SKG_OK;
  skg_status_t st = check_inputs(m, n, k, A, lda, B, ldb, a_layout, b_layout);
  if (st != SKG_OK) return st;
  const int sms = sm_count_cached();
  if (sms <= 0) return SKG_ERR_CUDA;
  skg_opts_t forced;
  if (opts) forced = *opts;
  else skg_opts_default(&forced);
  forced.abft = 1;
  Resolved r;
  st = resolve(m, n, k, &forced, r, sms);
  if (st != SKG_OK) return st;
  const Layout L = layout(m, n, k, r);
  if (!workspace || !aligned16(workspace) || ws_bytes < L.total) return SKG_ERR_WORKSPACE;
  if (!tensor_map_encoder()) return SKG_ERR_CUDA;
  uint8_t* ws = (uint8_t*)workspace;
  return run_encode_layouts(in_dtype, A, lda, a_layout == SKG_A_COL, m, B, ldb,
                            b_layout == SKG_B_NMAJOR, n, k, r, ws, L, sms, (cudaStream_t)stream);
}

skg_status_t skg_schedule_query(int64_t m, int64_t n, int64_t k, int32_t bm, int32_t bn,
                                int32_t bk, int32_t g, int32_t sched, skg_segment_t* out,
                                int64_t cap, int64_t* n_out) {
  if (m < 0 || n < 0 || k < 0 || bm <= 0 || bn <= 0 || bk <= 0 || g <= 0 || !n_out)
    return SKG_ERR_ARG;
  if (sched < SKG_SCHED_DP || sched > SKG_SCHED_SK2_DP) return SKG_ERR_ARG;
  if (cap > 0 && !out) return SKG_ERR_ARG;
  const Schedule s = make_schedule(m, n, k, bm, bn, bk, g, sched);
  int64_t count = 0;
  if (s.t > 0 && s.ipt > 0) {
    for (int x = 0; x < g; ++x) {
      Cursor c;
      c.init(s, x);
      Work w;
      while (c.next(s, w)) {
        if (count < cap) {
          out[count].cta = x;
          out[count].tile = w.tile;
          out[count].k_iter_begin = w.kb_begin;
          out[count].k_iter_end = w.kb_end;
          out[count].role = w.role;
        }
        ++count;
      }
    }
  }
  *n_out = count;
  return SKG_OK;
}

skg_status_t skg_schedule_cost(int64_t m, int64_t n, int64_t k, int32_t bm, int32_t bn,
                               int32_t bk, int32_t g, int32_t sched, double* us) {
  if (m < 0 || n < 0 || k < 0 || g <= 0 || !us) return SKG_ERR_ARG;
  if (bm != kTileM || bk != kTileK || (bn != 64 && bn != 128 && bn != 256))
    return SKG_ERR_UNSUPPORTED;
  if (sched < SKG_SCHED_DP || sched > SKG_SCHED_SK2_DP) return SKG_ERR_ARG;
  const Schedule s = make_schedule(m, n, k, bm, bn, bk, g, sched);
  *us = predict_us(s, model_for(bn), true);
  return SKG_OK;
}

skg_status_t skg_launch_shape(int64_t m, int64_t n, int64_t k, const skg_opts_t* opts,
                              int32_t* tile_n, int32_t* grid, int32_t* sched) {
  if (m < 0 || n < 0 || k < 0) return SKG_ERR_ARG;
  Resolved r;
  const int sms = sm_count_cached();
  skg_status_t st = resolve(m, n, k, opts, r, sms);
  if (st != SKG_OK) return st;
  if (r.abft && !r.abft_local && !r.ilc && m > 0 && n > 0 && k > 0 &&
      can_fuse_checksums(layout(m, n, k, r), r.bn))
    plan_fused(m, n, opts, SKG_IN_BF16, true, r);
  if (tile_n) *tile_n = r.bn;
  if (grid) *grid = r.grid + r.grid_ck;
  if (sched) *sched = r.sched;
  return SKG_OK;
}

skg_status_t skg_launch_plan(int64_t m, int64_t n, int64_t k, const skg_opts_t* opts,
                             skg_plan_t* out) {
  if (m < 0 || n < 0 || k < 0 || !out) return SKG_ERR_ARG;
  Resolved r;
  const int sms = sm_count_cached();
  skg_status_t st = resolve(m, n, k, opts, r, sms);
  if (st != SKG_OK) return st;
  const bool fused = r.abft && !r.abft_local && !r.ilc && m > 0 && n > 0 && k > 0 &&
                     can_fuse_checksums(layout(m, n, k, r), r.bn);
  if (fused) plan_fused(m, n, opts, SKG_IN_BF16, true, r);
  memset(out, 0, sizeof(*out));
  out->tile_m = r.pair ? 2 * kBM : kBM;
  out->tile_n = r.bn;
  out->ctas = r.grid;
  out->cta_pair = r.pair ? 2 : 1;
  out->sched = r.sched;
  out->side_ctas = fused ? r.grid_ck : 0;
  out->side_checksum_ctas = fused ? (r.grid_ck ? r.grid_ckt : 0) : 0;
  out->fused_checksums = fused ? 1 : 0;
  out->encode_in_kernel = r.enc_inkernel;
  out->local_checksums = r.abft_local;
  out->inloop_checksums = r.ilc;
  return SKG_OK;
}

skg_status_t skg_report_read(const void* workspace, skg_report_t* out, int32_t reset,
                             void* stream) {
  if (!workspace || !out) return SKG_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SKG_ERR_CUDA;
  const uint8_t* rep = (const uint8_t*)workspace + 256;
  if (cudaMemcpy(out, rep, sizeof(skg_report_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SKG_ERR_CUDA;
  if (reset) {
    if (cudaMemsetAsync((void*)rep, 0, sizeof(skg_report_t), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return SKG_ERR_CUDA;
  }
  return SKG_OK;
}

size_t skg_host_staging_size(int64_t m, int64_t n, int64_t k, int32_t in_dtype,
                             int32_t out_dtype, int32_t a_layout, int32_t b_layout) {
  Staging S;
  return staging_plan(m, n, k, in_dtype, out_dtype, a_layout, b_layout, S) ? S.total : 0;
}

skg_status_t skg_gemm_host(int64_t m, int64_t n, int64_t k, float alpha, const void* A,
                           int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                           int64_t ldc, int32_t in_dtype, int32_t out_dtype, int32_t a_layout,
                           int32_t b_layout, const skg_opts_t* opts, void* staging,
                           size_t staging_bytes, void* workspace, size_t ws_bytes,
                           void* stream_v) {
  Staging S;
  if (!staging_plan(m, n, k, in_dtype, out_dtype, a_layout, b_layout, S)) return SKG_ERR_ARG;
  if (m == 0 || n == 0) return SKG_OK;
  if (!C || ldc < n) return SKG_ERR_ARG;
  if (k > 0 && (!A || !B || lda < S.a_cols || ldb < S.b_cols)) return SKG_ERR_ARG;
  if (!staging || !aligned16(staging) || staging_bytes < S.total) return SKG_ERR_WORKSPACE;
  cudaStream_t stream = (cudaStream_t)stream_v;
  uint8_t* sb = (uint8_t*)staging;
  const int ob = S.out_bytes;
  if (k > 0) {
    if (cudaMemcpy2DAsync(sb + S.a, (size_t)S.lda * 2, A, (size_t)lda * 2, (size_t)S.a_cols * 2,
                          (size_t)S.a_rows, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpy2DAsync(sb + S.b, (size_t)S.ldb * 2, B, (size_t)ldb * 2, (size_t)S.b_cols * 2,
                          (size_t)S.b_rows, cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return SKG_ERR_CUDA;
  }
  if (beta != 0.f &&
      cudaMemcpy2DAsync(sb + S.c, (size_t)S.ldc * ob, C, (size_t)ldc * ob, (size_t)n * ob,
                        (size_t)m, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return SKG_ERR_CUDA;
  const skg_status_t st = gemm_impl(m, n, k, alpha, sb + S.a, S.lda, sb + S.b, S.ldb, beta,
                                    sb + S.c, S.ldc, in_dtype, out_dtype, a_layout, b_layout,
                                    opts, 0, workspace, ws_bytes, stream);
  if (st != SKG_OK) return st;
  return cudaMemcpy2DAsync(C, (size_t)ldc * ob, sb + S.c, (size_t)S.ldc * ob, (size_t)n * ob,
                           (size_t)m, cudaMemcpyDeviceToHost, stream) == cudaSuccess
             ? SKG_OK
             : SKG_ERR_CUDA;
}

int32_t skg_device_sm_count(void) { return sm_count_cached(); }

const char* skg_status_string(int32_t status) {
  switch (status) {
    case SKG_OK: return "ok";
    case SKG_ERR_ARG: return "invalid argument";
    case SKG_ERR_UNSUPPORTED: return "unsupported shape, layout or alignment";
    case SKG_ERR_CUDA: return "CUDA error";
    case SKG_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SKG_ERR_FIXUP_TIMEOUT: return "Stream-K fixup wait timed out";
    case SKG_ERR_PIPELINE_TIMEOUT: return "pipeline wait timed out";
    case SKG_ABFT_CORRECTED: return "ABFT: single fault located and corrected";
    case SKG_ABFT_UNCORRECTABLE: return "ABFT: uncorrectable checksum mismatch";
    default: return "unknown status";
  }
}

}  // extern "C"
