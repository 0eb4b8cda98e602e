// C ABI entry points: argument validation, the dispatch heuristic and kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "qgemm.h"
#include "kernels.h"
#include "qgemm_internal.h"

using namespace qgemm;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kSplitMaxM = 1024;          // split-K is considered only up to this M
// Above kSplitMaxM, stream-K over the leftover tiles is considered for K of at least this
// many 128-K blocks, where a cut piece is long enough to pay for its partial-tile store and
// read-back (measured with 256-token tiles: 8192 x 28672 at M = 1536 / 2048: -6 / -7%;
// 4096 x 7168 at M = 4096: +15% BF16, +41% FP8).
constexpr int64_t kSkLongKBlocks = 128;
constexpr uint64_t kTimeoutNs = 4000000000ull;     // default limit of one device wait

int g_debug_skip_first_x = 0;
uint64_t g_debug_timeout_ns = 0;

// Limit of every bounded wait inside a kernel: QGEMM_TIMEOUT_MS in the environment (read
// once; a profiler that replays each launch many times needs a longer limit), else 4 s;
// qgemm_debug_stall may override it.
uint64_t timeout_ns() {
  if (g_debug_timeout_ns != 0) return g_debug_timeout_ns;
  static const uint64_t v = []() -> uint64_t {
    const char* e = std::getenv("QGEMM_TIMEOUT_MS");
    if (e != nullptr) {
      char* end = nullptr;
      const unsigned long long ms = std::strtoull(e, &end, 10);
      if (end != e && ms > 0 && ms < 86400000ull) return uint64_t(ms) * 1000000ull;
    }
    return kTimeoutNs;
  }();
  return v;
}

struct DeviceInfo {
  bool init = false;
  bool ok = false;
  int sms = 0;
  int64_t l2_bytes = 0;
  int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;
int g_force_tile = 0;
int g_force_splits = 0;

bool current_device(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    d.init = true;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    d.l2_bytes = l2 > 0 ? l2 : (64ll << 20);
    d.status = device_status_ptr();
    d.ok = (major == 10 && minor == 3) && d.sms > 0 && d.status != nullptr;
  }
  *out = &d;
  return d.ok;
}

int sms_or_default() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
    return sms;
  return 152;
}

bool layout_of(const qgemm_wdesc* d, Layout* L) {
  if (d == nullptr || (d->flags & ~QGEMM_FLAG_BATCH_INVARIANT) != 0) return false;
  return make_layout(d->wfmt, d->sdtype, d->group_size, d->has_zp, d->afmt, d->N, d->K, L);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// FP4-operand records are addressed by a 32-bit tensor coordinate.
bool fp4_operand_records_fit(const Layout& L) {
  return L.afmt != A_FP8N || L.n_tiles * L.k_blocks < (int64_t(1) << 31);
}

// ---------------------------------------------------------------- dispatch
// Token tile and schedule from a cost model of one call on a persistent grid of P CTAs.
// Schedules (T = m_tiles * n_tiles tiles of k_blocks 128-K records each):
//   uniform  every tile cut into s equal K parts (s = 1: plain data-parallel), unit u on
//            CTA u % P: time ~ T0 + ceil(T s / P) (ceil(k_blocks / s) stage + unit
//                                                  + [s > 1] (reduce + s tile reduce))
//   stream-K the records of the T mod P leftover tiles (all T when T < P) are dealt out
//            evenly over the P CTAs, which then take the remaining whole tiles:
//            time ~ T0 + (records per CTA) stage + (units per CTA) unit
//                       + [no whole tiles] contributors tile reduce
// (stream-K, after "Stream-K: Work-centric Parallel Decomposition for Dense Matrix-Matrix
// Multiplication on the GPU", Osama et al., 2023: the cut pieces run first, so their
// reduction overlaps the whole tiles that follow).
namespace {
constexpr int kTiles[5] = {16, 32, 64, 128, 256};
constexpr double kStageUs[5] = {0.326, 0.330, 0.353, 0.401, 0.657};  // per 128-K block
constexpr double kUnitUs[5] = {3.08, 6.11, 7.88, 10.05, 17.59};      // per unit
constexpr double kReduceUsPerSplitRow = 0.0716;
// A cut tile's last contributor also waits for the others' partial tiles and reads them
// back from L2: 1 to 1.5 us more than a whole tile's epilogue (per-CTA timestamps of
// 16-token tiles cut in two).
constexpr double kReduceFixedUs = 1.0;
constexpr double kCallUs = 6.44;
constexpr int kMaxContrib = 8;       // stream-K (unforced): at most this many CTAs per tile
}  // namespace

// The CTA whose stream-K range holds record x of S (same formula as the kernel).
int64_t sk_cta_of(int64_t x, int64_t S, int64_t P) { return ((x + 1) * P - 1) / S; }

struct SkShape {
  int sk_tiles = 0, max_contrib = 0, max_units = 0;
  int64_t max_records = 0;
};

// Stream-K over the leftover tiles for T tiles of kb records on P CTAs.
SkShape sk_shape(int64_t T, int64_t kb, int64_t P) {
  SkShape r;
  const int64_t q = T / P;
  r.sk_tiles = int(q == 0 ? T : T % P);
  if (r.sk_tiles == 0) return r;
  const int64_t S = int64_t(r.sk_tiles) * kb;
  // CTAs holding a record of tile t: first..last when every CTA holds one (S >= P); with
  // fewer records than CTAs each CTA holds at most one, so a tile has kb contributors.
  for (int64_t t = 0; t < r.sk_tiles; ++t) {
    const int64_t c = S >= P ? sk_cta_of((t + 1) * kb - 1, S, P) - sk_cta_of(t * kb, S, P) + 1
                             : kb;
    r.max_contrib = std::max<int>(r.max_contrib, int(c));
  }
  for (int64_t i = 0; i < P; ++i) {
    const int64_t lo = i * S / P, hi = (i + 1) * S / P;
    const int64_t pieces = hi > lo ? (hi - 1) / kb - lo / kb + 1 : 0;
    r.max_units = std::max<int>(r.max_units, int(q + pieces));
    r.max_records = std::max<int64_t>(r.max_records, q * kb + (hi - lo));
  }
  if (r.max_contrib <= 1) r.max_contrib = 0;      // nothing is cut
  return r;
}

double plan_cost_us(const Layout& L, int64_t M, int ti, int splits, int sms) {
  const int64_t tt = kTiles[ti];
  const int64_t m_tiles = (M + tt - 1) / tt;
  const int64_t units = m_tiles * L.n_tiles * splits;
  const int64_t per_cta = (units + sms - 1) / sms;
  const int64_t kpu = (L.k_blocks + splits - 1) / splits;
  double unit = double(kpu) * kStageUs[ti] + kUnitUs[ti];
  if (splits > 1) unit += kReduceFixedUs + double(splits) * double(tt) * kReduceUsPerSplitRow;
  return kCallUs + double(per_cta) * unit;
}

// The kernel's stream-K arithmetic is 32-bit: (record + 1) * SMs must stay below 2^32 for
// the fewer than SMs cut tiles (a limit far above practical K).
bool sk_fits(const Layout& L, int sms) {
  return uint64_t(sms) * uint64_t(sms) * uint64_t(L.k_blocks) < (uint64_t(1) << 32);
}

double sk_cost_us(const Layout& L, int64_t M, int ti, int sms, SkShape* out) {
  *out = SkShape();
  if (!sk_fits(L, sms)) return 1e300;
  const int64_t tt = kTiles[ti];
  const int64_t T = (M + tt - 1) / tt * L.n_tiles;
  const SkShape sh = sk_shape(T, L.k_blocks, sms);
  *out = sh;
  if (sh.sk_tiles == 0 || (sh.max_contrib > kMaxContrib && g_force_splits >= 0)) return 1e300;
  double c = kCallUs + double(sh.max_records) * kStageUs[ti] + double(sh.max_units) * kUnitUs[ti];
  if (T < sms) c += kReduceFixedUs + double(sh.max_contrib) * double(tt) * kReduceUsPerSplitRow;
  return c;
}

bool batch_invariant(const qgemm_wdesc* d) { return (d->flags & QGEMM_FLAG_BATCH_INVARIANT) != 0; }

// The one schedule of batch-invariant calls: 128-token tiles (one MMA issuer, so a tile's
// stages accumulate in K order into one accumulator), no cut, no stream-K.
constexpr int kInvariantTile = 128;

// large_m_sk = false leaves out stream-K above kSplitMaxM (for a workspace that cannot hold
// its partial tiles).
GemmPlan plan_dense(const Layout& L, int64_t M, int sms, bool invariant = false,
                    bool large_m_sk = true) {
  GemmPlan p;
  p.token_tile = 16;
  p.splits = 1;
  p.sk_tiles = 0;
  p.max_contrib = 0;
  if (invariant) {
    p.token_tile = kInvariantTile;
    p.grid = int(std::min<int64_t>((M + kInvariantTile - 1) / kInvariantTile * L.n_tiles, sms));
    return p;
  }
  double best = 1e300;
  for (int ti = 0; ti < 5; ++ti) {
    const int tt = kTiles[ti];
    if (g_force_tile ? tt != g_force_tile : (tt > 16 && tt > 2 * M)) continue;
    if (g_force_splits >= 0) {
      for (int s : {1, 2, 3, 4, 6, 8}) {
        if (g_force_splits > 0) {
          if (s != 1) break;
          s = int(std::min<int64_t>(g_force_splits, L.k_blocks));
        } else if (s > 1 && (M > kSplitMaxM || L.k_blocks / s < 2)) {
          break;
        }
        const double c = plan_cost_us(L, M, ti, s, sms);
        if (c < best) {
          best = c;
          p.token_tile = tt;
          p.splits = s;
          p.sk_tiles = 0;
          p.max_contrib = s > 1 ? s : 0;
        }
        if (g_force_splits > 0) break;
      }
    }
    if (g_force_splits <= 0 &&
        (M <= kSplitMaxM || (large_m_sk && L.k_blocks >= kSkLongKBlocks))) {
      SkShape sh;
      const double c = sk_cost_us(L, M, ti, sms, &sh);
      if (c < best) {
        best = c;
        p.token_tile = tt;
        p.splits = 1;
        p.sk_tiles = sh.sk_tiles;
        p.max_contrib = sh.max_contrib;
      }
    }
  }
  if (g_force_tile) p.token_tile = g_force_tile;
  const int64_t tiles = (M + p.token_tile - 1) / p.token_tile * L.n_tiles;
  p.grid = p.sk_tiles > 0 ? sms : int(std::min<int64_t>(tiles * p.splits, sms));
  return p;
}

// Partial-sum slots and arrival counters of the cut tiles: a uniform cut of s parts needs
// s slots per tile, stream-K fewer than sk_tiles + grid slots (see the kernel's unit_at).
void cut_sizes(const Layout& L, int64_t M, const GemmPlan& p, int64_t* slots, int64_t* counters) {
  *slots = *counters = 0;
  if (p.sk_tiles > 0) {
    if (p.max_contrib == 0) return;
    *slots = p.sk_tiles + p.grid;
    *counters = p.sk_tiles;
  } else if (p.splits > 1) {
    *counters = (M + p.token_tile - 1) / p.token_tile * L.n_tiles;
    *slots = *counters * p.splits;
  }
}

int64_t slot_bytes(int token_tile) { return int64_t(kTileN) * token_tile * 4; }

int64_t split_ws_bytes(const Layout& L, int64_t M, const GemmPlan& p) {
  int64_t slots, counters;
  cut_sizes(L, M, p, &slots, &counters);
  if (slots == 0) return 0;
  return slots * slot_bytes(p.token_tile) + round_up(counters * 4, 256);
}

// Stream-K above kSplitMaxM runs only when the workspace (`avail` bytes) holds its partial
// tiles after the FP16 activation copy; otherwise the call keeps whole tiles.
bool large_m_sk_fits(const Layout& L, int64_t M, const GemmPlan& p, int64_t avail) {
  if (M <= kSplitMaxM || p.sk_tiles == 0) return true;
  const int64_t copy = f16_operands(L) ? prep_x_f16_bytes(M, L.K) : 0;
  return copy + split_ws_bytes(L, M, p) <= avail;
}

// MoE: the token tile from the average rows per expert (padding included); the stream-K
// workspace holds 2 * SMs slots and SMs counters.  Every m-tile of an expert streams the
// expert's weights again, and an expert a little above a multiple of the tile pays for a
// nearly empty one, so 128-token tiles are kept up to 192 rows per expert (64 experts of
// MXFP4 4096 x 7168, top-2, at 131 rows per expert: 571 against 654 us with 256-token tiles,
// 696 against 875 skewed).  Above that the 256-token tiles' fewer weight re-reads win on
// experts with many rows: 256 experts, top-8, 259 rows per expert, skewed routing, gate_up
// 3536 against 3993 us and down 1947 against 2387 us; uniform down 1945 against 2107 us.
int moe_token_tile(int64_t R, int32_t E) {
  const int64_t avg = R / E;
  int tt = avg <= 16 ? 16 : avg <= 32 ? 32 : avg <= 64 ? 64 : avg <= 192 ? 128 : 256;
  if (g_force_tile) tt = g_force_tile;
  return tt;
}

// Indexed (gathered) MoE: the grouped rule, token tiles up to 64.
int moe_indexed_token_tile(int64_t R, int32_t E) {
  const int64_t avg = R / E;
  int tt = avg <= 16 ? 16 : avg <= 32 ? 32 : 64;
  if (g_force_tile) tt = g_force_tile;
  return tt;
}

int64_t moe_ws_bytes(int tt, int sms) {
  return 2 * int64_t(sms) * slot_bytes(tt) + round_up(int64_t(sms) * 4, 256);
}

// MXFP4 with BF16 activations: the calls that may run on FP16 operands (given the
// workspace for the activation copy), by their token tile; see mx_f16_capable().
bool mx_f16_call(const Layout& L, int token_tile, bool invariant) {
  return mx_f16_capable(L) && !invariant && token_tile <= kMxF16MaxTile;
}

// Indexed MoE over more than a few hundred rows: the rows gathered into the workspace in
// sorted order (and, for FP8 or FP16 activations, their scales) for the grouped kernel.
// The in-kernel gather shares the issue slots with the dequant warps; the separate gather
// costs one launch (256 experts of MXFP4 4096 x 7168, top-8: at 64 rows 48.8 against 41.0
// us, at 576 / 848 / 1808 / 2024 rows 10-14% faster than the in-kernel gather).
constexpr int64_t kIndexedCopyMinRows = 256;

int64_t indexed_copy_bytes(const Layout& L, int64_t R, bool fp8) {
  const int64_t esz = fp8 ? 1 : 2;
  return round_up(R * L.K * esz, 256) + round_up(R * 4, 256);   // rows, then their scales
}

typedef PFN_cuTensorMapEncodeTiled_v12000 EncodeFn;

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// The map of X the kernel loads with 128-byte swizzle (the layout the MMA's shared-memory
// descriptor expects).  When K is a whole number of 128-byte slabs, X is described as a
// 3-D tensor [K / slab][rows][slab] so that one load brings several slabs (several
// pipeline stages for narrow token tiles); otherwise as a 2-D tensor [rows][K] loaded one
// slab at a time.  Sets *is_3d accordingly.
enum XType { X_BF16 = 0, X_F16 = 1, X_FP8 = 2 };

bool make_x_map(CUtensorMap* m, const void* X, XType xt, int64_t rows, int64_t K, int64_t ldx,
                int box_rows, int* is_3d) {
  EncodeFn enc = encode_fn();
  if (enc == nullptr) return false;
  const bool fp8 = xt == X_FP8;
  const int esize = fp8 ? 1 : 2;
  const int64_t slab = 128 / esize;                        // elements per 128-byte slab
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : xt == X_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int box_slabs = gemm_x_box_slabs(fp8, box_rows);
  if (K % slab == 0 && box_slabs > 0) {
    cuuint64_t dims[3] = {cuuint64_t(slab), cuuint64_t(rows), cuuint64_t(K / slab)};
    cuuint64_t strides[2] = {cuuint64_t(ldx) * esize, 128};
    cuuint32_t box[3] = {cuuint32_t(slab), cuuint32_t(box_rows), cuuint32_t(box_slabs)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(m, dt, 3, const_cast<void*>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      *is_3d = 1;
      return true;
    }
  }
  cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(ldx) * esize};
  cuuint32_t box[2] = {cuuint32_t(slab), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(X), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  *is_3d = 0;
  return r == CUDA_SUCCESS;
}

// MXFP4 activation codes (W4A4): [rows][K / 2] bytes with row stride ldq bytes, loaded as
// 64-byte rows (128 K) with the 64-byte swizzle the FP4 MMA's descriptor expects.
bool make_x4_map(CUtensorMap* m, const void* Xq, int64_t rows, int64_t K, int64_t ldq,
                 int box_rows) {
  EncodeFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(K / 2), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(ldq)};
  cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(Xq), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 activations on FP4 operands: the packed codes of E experts as a 4-D tensor of 4-bit
// elements [E][records][128 rows][128], rows 64 bytes apart, records record_bytes and experts
// expert_stride bytes apart; a box is one record, which the TMA writes as 128-byte rows (16
// elements in the first 8 bytes of every 16) with the 128-byte swizzle.
bool make_w4_map(CUtensorMap* m, const Layout& L, const void* packed, int32_t E,
                 int64_t expert_stride) {
  EncodeFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {128, 128, cuuint64_t(L.n_tiles * L.k_blocks), cuuint64_t(E)};
  cuuint64_t strides[3] = {64, cuuint64_t(L.record_bytes), cuuint64_t(expert_stride)};
  cuuint32_t box[4] = {128, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  void* base = const_cast<uint8_t*>(static_cast<const uint8_t*>(packed) + kHeaderBytes);
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Exponent rows of MXFP4 activations: one byte per 32 K; the kernel loads them in 16-byte
// boxes (four 128-K blocks), so a row spans a whole number of boxes.
int64_t exps_row_min(int64_t K) { return round_up((K / 32 + 3) / 4 * 4, 16); }

// The exponents [rows][ld_exps] bytes for TMA: boxes of 16 bytes x box_rows rows.
bool make_exps_map(CUtensorMap* m, const void* exps, int64_t rows, int64_t ld_exps,
                   int box_rows) {
  EncodeFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cuuint64_t(ld_exps), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(ld_exps)};
  cuuint32_t box[2] = {16, cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(exps), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

qgemm_status check_x(const void* X, bool fp8, int64_t rows, int64_t K, int64_t ldx) {
  if (X == nullptr || rows < 0 || rows >= (int64_t(1) << 31) || ldx < K) return QGEMM_ERR_INVALID_ARG;
  if (!aligned(X, 16) || (ldx * (fp8 ? 1 : 2)) % 16 != 0) return QGEMM_ERR_ALIGNMENT;
  return QGEMM_OK;
}

// MXFP4 activations: codes [rows][ldq bytes] (ldq >= K / 2) and exponents [rows][lde].
qgemm_status check_x4(const void* Xq, int64_t rows, int64_t K, int64_t ldq, const void* exps,
                      int64_t lde) {
  if (Xq == nullptr || exps == nullptr || rows < 0 || rows >= (int64_t(1) << 31) ||
      ldq < K / 2 || lde < exps_row_min(K))
    return QGEMM_ERR_INVALID_ARG;
  if (!aligned(Xq, 16) || ldq % 16 != 0 || !aligned(exps, 16) || lde % 16 != 0)
    return QGEMM_ERR_ALIGNMENT;
  return QGEMM_OK;
}

qgemm_status check_y(const void* Y, int64_t N, int64_t ldy) {
  if (Y == nullptr || ldy < N) return QGEMM_ERR_INVALID_ARG;
  if (!aligned(Y, 2)) return QGEMM_ERR_ALIGNMENT;
  return QGEMM_OK;
}

// Every argument check of the dense calls that needs no device.
qgemm_status check_dense(const qgemm_wdesc* desc, int32_t afmt, const void* packed,
                         const void* X, int64_t M, int64_t ldx, const float* tok_scale,
                         const float* chan_scale, const float* bias, const void* Y, int64_t ldy,
                         Layout* L, const uint8_t* x_exps = nullptr, int64_t ld_exps = 0) {
  if (!layout_of(desc, L)) return QGEMM_ERR_INVALID_ARG;
  const bool fp8 = afmt == A_FP8;
  // FP8 activations run on either W4A8 packing: register-decoded or FP4 operands
  if (L->afmt != afmt && !(fp8 && L->afmt == A_FP8N)) return QGEMM_ERR_INVALID_ARG;
  if (!fp4_operand_records_fit(*L)) return QGEMM_ERR_UNSUPPORTED;
  if (fp8 && L->wfmt != W_MXFP4) return QGEMM_ERR_UNSUPPORTED;
  if (M < 0) return QGEMM_ERR_INVALID_ARG;
  if (packed == nullptr) return QGEMM_ERR_INVALID_ARG;
  if (!aligned(packed, 256)) return QGEMM_ERR_ALIGNMENT;
  qgemm_status s = afmt == A_MXFP4 ? check_x4(X, M, L->K, ldx, x_exps, ld_exps)
                                   : check_x(X, fp8, M, L->K, ldx);
  if (s != QGEMM_OK) return s;
  if ((s = check_y(Y, L->N, ldy)) != QGEMM_OK) return s;
  if (fp8 && tok_scale == nullptr) return QGEMM_ERR_INVALID_ARG;
  if ((chan_scale && !aligned(chan_scale, 4)) || (tok_scale && !aligned(tok_scale, 4)) ||
      (bias && !aligned(bias, 4)))
    return QGEMM_ERR_ALIGNMENT;
  return QGEMM_OK;
}

qgemm_status run_dense(const qgemm_wdesc* desc, int32_t afmt, const void* packed, const void* X,
                       int64_t M, int64_t ldx, const float* tok_scale, const float* chan_scale,
                       const float* bias, void* Y, int64_t ldy, void* ws, size_t ws_bytes,
                       void* stream, const uint8_t* x_exps = nullptr, int64_t ld_exps = 0) {
  Layout L;
  const qgemm_status s = check_dense(desc, afmt, packed, X, M, ldx, tok_scale, chan_scale, bias,
                                     Y, ldy, &L, x_exps, ld_exps);
  const bool fp8 = afmt == A_FP8, a4 = afmt == A_MXFP4;
  if (s != QGEMM_OK) return s;
  if (M == 0) return QGEMM_OK;
  DeviceInfo* dev = nullptr;
  if (!current_device(&dev)) return QGEMM_ERR_NO_DEVICE;
  GemmPlan plan = plan_dense(L, M, dev->sms, batch_invariant(desc));
  if (!large_m_sk_fits(L, M, plan, ws == nullptr ? 0 : int64_t(ws_bytes)))
    plan = plan_dense(L, M, dev->sms, batch_invariant(desc), false);
  // FP16 operands: the pre-pass's FP16 rows and row scales lead the workspace (INT4 with
  // BF16 scales always; MXFP4 in small calls when the workspace holds the copy)
  const int64_t split = split_ws_bytes(L, M, plan);
  const bool f16 = f16_operands(L) ||
                   (mx_f16_call(L, plan.token_tile, batch_invariant(desc)) && ws != nullptr &&
                    int64_t(ws_bytes) >= prep_x_f16_bytes(M, L.K) + split);
  plan.mx_f16 = f16 && !f16_operands(L);
  const int64_t prep = f16 ? prep_x_f16_bytes(M, L.K) : 0;
  const int64_t need = prep + split;
  if (need > 0 && (ws == nullptr || int64_t(ws_bytes) < need)) return QGEMM_ERR_WORKSPACE;
  if (need > 0 && !aligned(ws, 256)) return QGEMM_ERR_ALIGNMENT;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const void* xg = X;                                    // what the GEMM reads as X
  int64_t ldg = ldx;
  float* rowscale = nullptr;
  if (f16) {
    rowscale = reinterpret_cast<float*>(wsb + round_up(M * L.K * 2, 256));
    if (launch_prep_x_f16(X, M, L.K, ldx, wsb, rowscale, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return QGEMM_ERR_CUDA;
    xg = wsb;
    ldg = L.K;
    plan.pdl = 1;
  }
  CUtensorMap tmap;
  int x3d = 0;
  if (a4 ? !make_x4_map(&tmap, X, M, L.K, ldx, plan.token_tile)
         : !make_x_map(&tmap, xg, fp8 ? X_FP8 : f16 ? X_F16 : X_BF16, M, L.K, ldg,
                       plan.token_tile, &x3d))
    return QGEMM_ERR_CUDA;
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.x_3d = x3d;
  a.x_exps = x_exps;
  a.ld_exps = ld_exps;
  if (a4 && !make_exps_map(&a.tmap_e, x_exps, M, ld_exps, plan.token_tile)) return QGEMM_ERR_CUDA;
  if (L.afmt == A_FP8N && !make_w4_map(&a.tmap_w, L, packed, 1, L.total_bytes)) return QGEMM_ERR_CUDA;
  a.L = L;
  a.packed = static_cast<const uint8_t*>(packed);
  a.M = M;
  a.m_tiles = int((M + plan.token_tile - 1) / plan.token_tile);
  a.splits = plan.splits;
  a.num_units = plan.sk_tiles > 0 ? plan.grid : int(int64_t(a.m_tiles) * L.n_tiles * plan.splits);
  a.sk_tiles = plan.sk_tiles;
  // Token tiles per rasterization group: as many as keep the group's activation rows
  // within about half of L2, so that they are read from DRAM once.
  {
    const int64_t x_tile_bytes = int64_t(plan.token_tile) * (a4 ? L.K / 2 : L.K * (fp8 ? 1 : 2));
    const int64_t gm = std::max<int64_t>(1, (dev->l2_bytes / 2) / std::max<int64_t>(1, x_tile_bytes));
    a.group_m = int(std::min<int64_t>(gm, a.m_tiles));
  }
  a.chan_scale = chan_scale;
  a.bias = bias;
  a.tok_scale = f16 ? rowscale : tok_scale;
  a.Y = Y;
  a.ldy = ldy;
  if (need > prep) {
    int64_t slots, counters;
    cut_sizes(L, M, plan, &slots, &counters);
    a.ws = reinterpret_cast<float*>(wsb + prep);
    a.counters = reinterpret_cast<int32_t*>(wsb + prep + slots * slot_bytes(plan.token_tile));
  }
  a.status = dev->status;
  a.timeout_ns = timeout_ns();
  a.debug_skip_first_x = g_debug_skip_first_x;
  cudaError_t e = launch_gemm(fp8, plan, tmap, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QGEMM_OK : QGEMM_ERR_CUDA;
}

}  // namespace

namespace qgemm {

qgemm_status dense_a16_scratch(const qgemm_wdesc* desc, const void* packed, const void* X,
                               int64_t M, int64_t ldx, const float* chan_scale, const void* Y,
                               int64_t ldy, int64_t capacity, int64_t* need,
                               int64_t* counter_off, int64_t* counter_bytes) {
  *need = *counter_off = *counter_bytes = 0;
  Layout L;
  const qgemm_status s = check_dense(desc, A_BF16, packed, X, M, ldx, nullptr, chan_scale,
                                     nullptr, Y, ldy, &L);
  if (s != QGEMM_OK || M == 0) return s;
  DeviceInfo* dev = nullptr;
  if (!current_device(&dev)) return QGEMM_ERR_NO_DEVICE;
  GemmPlan plan = plan_dense(L, M, dev->sms, batch_invariant(desc));
  if (!large_m_sk_fits(L, M, plan, capacity))
    plan = plan_dense(L, M, dev->sms, batch_invariant(desc), false);
  int64_t slots, counters;
  cut_sizes(L, M, plan, &slots, &counters);
  const int64_t split = split_ws_bytes(L, M, plan);
  // the same choice as run_dense makes with a workspace of `need` bytes: INT4 with BF16
  // scales always takes the activation copy, small MXFP4 calls when it fits the capacity
  const bool f16 = f16_operands(L) ||
                   (mx_f16_call(L, plan.token_tile, batch_invariant(desc)) &&
                    prep_x_f16_bytes(M, L.K) + split <= capacity);
  const int64_t prep = f16 ? prep_x_f16_bytes(M, L.K) : 0;
  *need = prep + split;
  if (split > 0) {
    *counter_off = prep + slots * slot_bytes(plan.token_tile);
    *counter_bytes = split - slots * slot_bytes(plan.token_tile);
  }
  return QGEMM_OK;
}

}  // namespace qgemm

extern "C" {

int32_t qgemm_version(void) { return 100; }

const char* qgemm_status_str(qgemm_status s) {
  switch (s) {
    case QGEMM_OK: return "ok";
    case QGEMM_ERR_INVALID_ARG: return "invalid argument";
    case QGEMM_ERR_UNSUPPORTED: return "unsupported combination";
    case QGEMM_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case QGEMM_ERR_WORKSPACE: return "workspace missing or too small";
    case QGEMM_ERR_BAD_PACKED: return "packed weights do not match the descriptor";
    case QGEMM_ERR_CUDA: return "CUDA error";
    case QGEMM_ERR_TIMEOUT: return "device wait timed out";
    case QGEMM_ERR_NO_DEVICE: return "no sm_103 device is current";
    case QGEMM_ERR_BAD_VALUE: return "invalid value in weights, scales, zero points or offsets";
  }
  return "unknown status";
}

qgemm_status qgemm_check_desc(const qgemm_wdesc* desc) {
  Layout L;
  return layout_of(desc, &L) ? QGEMM_OK : QGEMM_ERR_INVALID_ARG;
}

size_t qgemm_packed_bytes(const qgemm_wdesc* desc) {
  Layout L;
  if (!layout_of(desc, &L)) return 0;
  return size_t(L.total_bytes);
}

qgemm_status qgemm_repack(const qgemm_wdesc* desc, const uint8_t* codes, const void* scales,
                          const uint8_t* zeros, void* packed, void* stream) {
  return qgemm_repack_scaled(desc, codes, scales, zeros, 1.0f, packed, stream);
}

qgemm_status qgemm_repack_scaled(const qgemm_wdesc* desc, const uint8_t* codes,
                                 const void* scales, const uint8_t* zeros, float global_scale,
                                 void* packed, void* stream) {
  Layout L;
  if (!layout_of(desc, &L)) return QGEMM_ERR_INVALID_ARG;
  // NVFP4's decode leaves the weights 2^8 smaller (e2m1 x s x 2^-8, exact in BF16): the
  // accumulators take 2^8 back with the per-tensor scale.  Other formats have none.
  const float acc_scale = L.wfmt == W_NVFP4 ? global_scale * 256.0f : global_scale;
  if (!std::isfinite(acc_scale)) return QGEMM_ERR_INVALID_ARG;
  if (L.wfmt != W_NVFP4 && global_scale != 1.0f) return QGEMM_ERR_UNSUPPORTED;
  if (codes == nullptr || scales == nullptr || packed == nullptr) return QGEMM_ERR_INVALID_ARG;
  if (L.has_zp && zeros == nullptr) return QGEMM_ERR_INVALID_ARG;
  if (!aligned(codes, 4) || !aligned(scales, L.scale_bytes) || !aligned(packed, 256))
    return QGEMM_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  if (!current_device(&dev)) return QGEMM_ERR_NO_DEVICE;
  cudaError_t e = launch_repack(L, codes, scales, L.has_zp ? zeros : nullptr, acc_scale, packed,
                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QGEMM_OK : QGEMM_ERR_CUDA;
}

size_t qgemm_workspace_bytes(const qgemm_wdesc* desc, int64_t M_max) {
  Layout L;
  if (!layout_of(desc, &L) || M_max <= 0) return 0;
  const int sms = sms_or_default();
  int64_t best = 0;
  const int64_t top = std::min<int64_t>(M_max, kSplitMaxM);
  const bool inv = batch_invariant(desc);
  // (MXFP4: narrow-tile calls also hold their FP16 activation copy)
  auto need = [&](int64_t M) {
    const GemmPlan p = plan_dense(L, M, sms, inv);
    return split_ws_bytes(L, M, p) + (mx_f16_call(L, p.token_tile, inv) ? prep_x_f16_bytes(M, L.K) : 0);
  };
  for (int64_t M = 1; M <= top; ++M) best = std::max(best, need(M));
  // Above kSplitMaxM a plan depends on M only through the tile counts ceil(M / tile), which
  // are the same for the 16 values of M up to each multiple of 16.
  if (L.k_blocks >= kSkLongKBlocks)
    for (int64_t M = kSplitMaxM + 16; M < M_max; M += 16) best = std::max(best, need(M));
  best = std::max(best, need(M_max));
  // FP16 operands (INT4 with BF16 scales): the activation copy, largest at M_max
  if (f16_operands(L)) best += prep_x_f16_bytes(M_max, L.K);
  return size_t(best);
}

qgemm_status qgemm_w4a16(const qgemm_wdesc* desc, const void* packed, const void* X, int64_t M,
                         int64_t ldx, const float* chan_scale, const float* bias, void* Y,
                         int64_t ldy, void* ws, size_t ws_bytes, void* stream) {
  return run_dense(desc, A_BF16, packed, X, M, ldx, nullptr, chan_scale, bias, Y, ldy, ws,
                   ws_bytes, stream);
}

qgemm_status qgemm_w4a8(const qgemm_wdesc* desc, const void* packed, const uint8_t* Xq, int64_t M,
                        int64_t ldx, const float* tok_scale, const float* chan_scale,
                        const float* bias, void* Y, int64_t ldy, void* ws, size_t ws_bytes,
                        void* stream) {
  return run_dense(desc, A_FP8, packed, Xq, M, ldx, tok_scale, chan_scale, bias, Y, ldy, ws,
                   ws_bytes, stream);
}

qgemm_status qgemm_w4a4(const qgemm_wdesc* desc, const void* packed, const uint8_t* Xq, int64_t M,
                        int64_t ldq, const uint8_t* x_exps, int64_t ld_exps,
                        const float* chan_scale, const float* bias, void* Y, int64_t ldy,
                        void* ws, size_t ws_bytes, void* stream) {
  return run_dense(desc, A_MXFP4, packed, Xq, M, ldq, nullptr, chan_scale, bias, Y, ldy, ws,
                   ws_bytes, stream, x_exps, ld_exps);
}

qgemm_status qgemm_quant_act_mxfp4(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                   int64_t ldq, uint8_t* x_exps, int64_t ld_exps, void* stream) {
  if (X == nullptr || Xq == nullptr || x_exps == nullptr || M < 0 || K < 32 || K % 32 != 0 ||
      ldx < K || ldq < K / 2 || ld_exps < exps_row_min(K) || M >= (int64_t(1) << 31))
    return QGEMM_ERR_INVALID_ARG;
  if (!aligned(X, 2) || !aligned(Xq, 4) || ldq % 4 != 0 || !aligned(x_exps, 16) ||
      ld_exps % 16 != 0)
    return QGEMM_ERR_ALIGNMENT;
  if (M == 0) return QGEMM_OK;
  DeviceInfo* dev = nullptr;
  if (!current_device(&dev)) return QGEMM_ERR_NO_DEVICE;
  cudaError_t e = launch_quant_act_mxfp4(X, M, K, ldx, Xq, ldq, x_exps, ld_exps,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QGEMM_OK : QGEMM_ERR_CUDA;
}

qgemm_status qgemm_quant_act_fp8(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                 int64_t ldq, float* tok_scale, void* stream) {
  if (X == nullptr || Xq == nullptr || tok_scale == nullptr || M < 0 || K < 1 || ldx < K ||
      ldq < K || M >= (int64_t(1) << 31))
    return QGEMM_ERR_INVALID_ARG;
  if (!aligned(X, 2) || !aligned(tok_scale, 4)) return QGEMM_ERR_ALIGNMENT;
  if (M == 0) return QGEMM_OK;
  DeviceInfo* dev = nullptr;
  if (!current_device(&dev)) return QGEMM_ERR_NO_DEVICE;
  cudaError_t e = launch_quant_act_fp8(X, M, K, ldx, Xq, ldq, tok_scale,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QGEMM_OK : QGEMM_ERR_CUDA;
}

}  // extern "C"

namespace {

// The grouped and the indexed MoE call: X has x_rows rows; row_index == nullptr means the
// rows are already sorted by expert (sorted position r is X row r).
qgemm_status run_moe(const qgemm_wdesc* desc, const void* packed, int32_t E, int32_t afmt,
                     const void* X, int64_t x_rows, int64_t ldx, const float* tok_scale,
                     const float* bias, const int32_t* expert_offsets, const int32_t* row_index,
                     int64_t R, void* Y, int64_t ldy, void* ws, size_t ws_bytes, void* stream) {
  Layout L;
  if (!layout_of(desc, &L)) return QGEMM_ERR_INVALID_ARG;
  const bool fp8 = afmt == QGEMM_A_FP8E4M3_TOKEN;
  if (afmt != QGEMM_A_BF16 && !fp8) return QGEMM_ERR_INVALID_ARG;
  if (L.afmt != afmt && !(fp8 && L.afmt == A_FP8N)) return QGEMM_ERR_INVALID_ARG;
  if (!fp4_operand_records_fit(L)) return QGEMM_ERR_UNSUPPORTED;
  if (E < 1 || E > 1024 || packed == nullptr || expert_offsets == nullptr || R < 0 || x_rows < 0)
    return QGEMM_ERR_INVALID_ARG;
  if (row_index != nullptr && R > 0 && x_rows == 0) return QGEMM_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(expert_offsets, 4) || !aligned(row_index, 4) ||
      !aligned(bias, 4))
    return QGEMM_ERR_ALIGNMENT;
  qgemm_status s = check_x(X, fp8, x_rows, L.K, ldx);
  if (s != QGEMM_OK) return s;
  if ((s = check_y(Y, L.N, ldy)) != QGEMM_OK) return s;
  if (fp8 && tok_scale == nullptr) return QGEMM_ERR_INVALID_ARG;
  if (R == 0) return QGEMM_OK;
  DeviceInfo* dev = nullptr;
  if (!current_device(&dev)) return QGEMM_ERR_NO_DEVICE;
  GemmPlan plan;
  const bool inv = batch_invariant(desc);
  if (inv && row_index != nullptr) return QGEMM_ERR_UNSUPPORTED;
  // FP16 operands: the pre-pass's FP16 copy of the x_rows rows of X and their row scales
  // lead the workspace, which is then required (INT4 with BF16 scales); MXFP4 experts take
  // them for narrow token tiles when the workspace holds the copy
  const bool mx = !fp8 && mx_f16_call(L, moe_token_tile(R, E), inv) && ws != nullptr &&
                  int64_t(ws_bytes) >= prep_x_f16_bytes(x_rows, L.K);
  const bool f16 = f16_operands(L) || mx;
  plan.mx_f16 = mx ? 1 : 0;
  const int64_t prep = f16 ? prep_x_f16_bytes(x_rows, L.K) : 0;
  if (f16 && (ws == nullptr || int64_t(ws_bytes) < prep)) return QGEMM_ERR_WORKSPACE;
  if ((f16 || ws != nullptr) && !aligned(ws, 256)) return QGEMM_ERR_ALIGNMENT;
  // Indexed calls over many rows gather them into the workspace first and run the grouped
  // kernel on the sorted copy, when the workspace holds it.
  const bool copy = row_index != nullptr && R >= kIndexedCopyMinRows &&
                    int64_t(ws_bytes) >= prep + indexed_copy_bytes(L, R, fp8) && g_force_tile == 0;
  const bool gather = row_index != nullptr && !copy;     // the gathering kernel
  const int tt = inv ? kInvariantTile : gather ? moe_indexed_token_tile(R, E) : moe_token_tile(R, E);
  if (gather && tt > 64) return QGEMM_ERR_UNSUPPORTED;   // gathering kernels: <= 64
  plan.token_tile = tt;
  plan.splits = 1;
  plan.sk_tiles = 0;
  plan.max_contrib = 0;
  plan.grid = dev->sms;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* xg = X;
  int64_t ldg = ldx;
  const float* tok = tok_scale;
  if (f16) {
    float* rowscale = reinterpret_cast<float*>(wsb + round_up(x_rows * L.K * 2, 256));
    if (launch_prep_x_f16(X, x_rows, L.K, ldx, wsb, rowscale, st) != cudaSuccess)
      return QGEMM_ERR_CUDA;
    xg = wsb;
    ldg = L.K;
    tok = rowscale;
    plan.pdl = 1;
  }
  int64_t head = prep;                                   // workspace bytes before the slots
  if (copy) {
    const int64_t esz = fp8 ? 1 : 2;
    uint8_t* sorted = wsb + prep;
    float* sorted_scale = (fp8 || f16) ? reinterpret_cast<float*>(sorted + round_up(R * L.K * esz, 256))
                                       : nullptr;
    if (launch_gather_rows(xg, ldg * esz, x_rows, row_index, R, L.K * esz, sorted, L.K * esz,
                           tok, sorted_scale, dev->status, st) != cudaSuccess)
      return QGEMM_ERR_CUDA;
    xg = sorted;
    ldg = L.K;
    tok = sorted_scale;
    plan.pdl = 0;                      // the GEMM follows the gather, not the pre-pass
    head += indexed_copy_bytes(L, R, fp8);
  }
  // the gathering kernel copies X rows itself and never reads a tensor map
  CUtensorMap tmap;
  memset(&tmap, 0, sizeof(tmap));
  int x3d = 0;
  if (!gather && !make_x_map(&tmap, xg, fp8 ? X_FP8 : f16 ? X_F16 : X_BF16, R, L.K, ldg, tt, &x3d))
    return QGEMM_ERR_CUDA;
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  if (gather) {
    a.x = static_cast<const uint8_t*>(xg);
    a.ldx_bytes = ldg * (fp8 ? 1 : 2);
    a.x_rows = x_rows;
  }
  a.x_3d = x3d;
  a.L = L;
  a.packed = static_cast<const uint8_t*>(packed);
  a.expert_stride = L.total_bytes;
  if (L.afmt == A_FP8N && !make_w4_map(&a.tmap_w, L, packed, E, L.total_bytes)) return QGEMM_ERR_CUDA;
  a.offsets = expert_offsets;
  a.row_index = gather ? row_index : nullptr;
  a.E = E;
  a.M = R;
  a.splits = 1;
  a.bias = bias;
  a.bias_stride = L.N;
  a.tok_scale = tok;
  a.Y = Y;
  a.ldy = ldy;
  // Stream-K needs the whole bound after the activation copies; a smaller (or no)
  // workspace keeps whole tiles.
  if (ws != nullptr && !inv && g_force_splits != 1 && sk_fits(L, plan.grid) &&
      int64_t(ws_bytes) >= head + moe_ws_bytes(tt, plan.grid)) {
    a.ws = reinterpret_cast<float*>(wsb + head);
    a.counters = reinterpret_cast<int32_t*>(wsb + head + 2 * int64_t(plan.grid) * slot_bytes(tt));
  }
  a.status = dev->status;
  a.timeout_ns = timeout_ns();
  cudaError_t e = launch_gemm(fp8, plan, tmap, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QGEMM_OK : QGEMM_ERR_CUDA;
}

}  // namespace

extern "C" {

qgemm_status qgemm_moe_grouped(const qgemm_wdesc* desc, const void* packed, int32_t E,
                               int32_t afmt, const void* X, int64_t R, int64_t ldx,
                               const float* tok_scale, const float* bias,
                               const int32_t* expert_offsets, void* Y, int64_t ldy, void* ws,
                               size_t ws_bytes, void* stream) {
  return run_moe(desc, packed, E, afmt, X, R, ldx, tok_scale, bias, expert_offsets, nullptr, R,
                 Y, ldy, ws, ws_bytes, stream);
}

qgemm_status qgemm_moe_indexed(const qgemm_wdesc* desc, const void* packed, int32_t E,
                               int32_t afmt, const void* X, int64_t T, int64_t ldx,
                               const float* tok_scale, const float* bias,
                               const int32_t* expert_offsets, const int32_t* row_index,
                               int64_t R, void* Y, int64_t ldy, void* ws, size_t ws_bytes,
                               void* stream) {
  if (row_index == nullptr && R > 0) return QGEMM_ERR_INVALID_ARG;
  return run_moe(desc, packed, E, afmt, X, T, ldx, tok_scale, bias, expert_offsets, row_index,
                 R, Y, ldy, ws, ws_bytes, stream);
}

size_t qgemm_act_copy_bytes(const qgemm_wdesc* desc, int64_t x_rows) {
  Layout L;
  if (!layout_of(desc, &L) || x_rows <= 0 || !f16_operands(L)) return 0;
  return size_t(prep_x_f16_bytes(x_rows, L.K));
}

size_t qgemm_moe_workspace_bytes(const qgemm_wdesc* desc, int32_t E, int64_t R) {
  Layout L;
  if (!layout_of(desc, &L) || E < 1 || R <= 0) return 0;
  const int tt = std::max(moe_token_tile(R, E), std::min(moe_indexed_token_tile(R, E), 64));
  const bool f16 = f16_operands(L) || mx_f16_call(L, moe_token_tile(R, E), false);
  const int64_t prep = f16 ? prep_x_f16_bytes(R, L.K) : 0;
  return size_t(prep + moe_ws_bytes(tt, sms_or_default()));
}

size_t qgemm_moe_indexed_workspace_bytes(const qgemm_wdesc* desc, int32_t E, int32_t afmt,
                                         int64_t T, int64_t R) {
  Layout L;
  if (!layout_of(desc, &L) || E < 1 || R <= 0 || T < 0) return 0;
  if (afmt != QGEMM_A_BF16 && afmt != QGEMM_A_FP8E4M3_TOKEN) return 0;
  const bool fp8 = afmt == QGEMM_A_FP8E4M3_TOKEN;
  const bool f16 = f16_operands(L) || (!fp8 && mx_f16_call(L, moe_token_tile(R, E), false));
  const int64_t prep = f16 ? prep_x_f16_bytes(T, L.K) : 0;
  const int64_t copy = R >= kIndexedCopyMinRows ? indexed_copy_bytes(L, R, fp8) : 0;
  const int tt = copy > 0 ? moe_token_tile(R, E) : std::min(moe_indexed_token_tile(R, E), 64);
  return size_t(prep + copy + moe_ws_bytes(tt, sms_or_default()));
}

qgemm_status qgemm_dequant_debug(const qgemm_wdesc* desc, const void* packed, void* W_out,
                                 void* stream) {
  Layout L;
  if (!layout_of(desc, &L)) return QGEMM_ERR_INVALID_ARG;
  if (packed == nullptr || W_out == nullptr) return QGEMM_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(W_out, 16)) return QGEMM_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  if (!current_device(&dev)) return QGEMM_ERR_NO_DEVICE;
  cudaError_t e = launch_dequant_debug(L, packed, W_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QGEMM_OK : QGEMM_ERR_CUDA;
}

qgemm_status qgemm_device_status(int32_t clear) {
  DeviceInfo* dev = nullptr;
  if (!current_device(&dev)) return QGEMM_ERR_NO_DEVICE;
  if (cudaDeviceSynchronize() != cudaSuccess) return QGEMM_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return QGEMM_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return QGEMM_ERR_CUDA;
  }
  return static_cast<qgemm_status>(v);
}

qgemm_status qgemm_plan(const qgemm_wdesc* desc, int64_t M, int32_t out[5]) {
  Layout L;
  if (!layout_of(desc, &L) || M <= 0 || out == nullptr) return QGEMM_ERR_INVALID_ARG;
  const GemmPlan p = plan_dense(L, M, sms_or_default(), batch_invariant(desc));
  out[0] = p.token_tile;
  out[1] = p.splits;
  out[2] = p.sk_tiles;
  out[3] = p.max_contrib;
  out[4] = p.grid;
  return QGEMM_OK;
}

qgemm_status qgemm_debug_stall(int32_t skip_first_x, int32_t timeout_ms) {
  if (skip_first_x < 0 || skip_first_x > 1 || timeout_ms < 0 || timeout_ms > 60000)
    return QGEMM_ERR_INVALID_ARG;
  g_debug_skip_first_x = skip_first_x;
  g_debug_timeout_ns = uint64_t(timeout_ms) * 1000000ull;
  return QGEMM_OK;
}

qgemm_status qgemm_force_config(int32_t token_tile, int32_t splits) {
  if (token_tile != 0 && token_tile != 16 && token_tile != 32 && token_tile != 64 &&
      token_tile != 128 && token_tile != 256)
    return QGEMM_ERR_INVALID_ARG;
  if (splits < -1 || splits > 64) return QGEMM_ERR_INVALID_ARG;
  g_force_tile = token_tile;
  g_force_splits = splits;
  return QGEMM_OK;
}

}  // extern "C"
