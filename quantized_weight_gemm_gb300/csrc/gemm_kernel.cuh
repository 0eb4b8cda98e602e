// The tcgen05 quantized-weight GEMM kernel (dense, MoE grouped and MoE indexed), sm_103a.
//
// One persistent CTA per SM, warp-specialised.  A "stage" is 128 K-elements of one work
// unit (a 128-row weight tile x a token tile, over a range of K); the 256-token BF16 variant
// uses half stages (64 K) so that its 32 KB activation tiles fit.  Warp roles, in order:
//
//   dequant     W warpgroups (4 for token tiles up to 64, else 2) taking the CTA's stages
//               round-robin: thread r owns weight row r (= tensor-memory lane r), decodes
//               its row's codes from the record ring in registers (dequant.cuh), releases
//               the record slot, and writes the weights with tcgen05.st into the stage's
//               A-operand columns of tensor memory.  The weights never touch shared memory.
//   epilogue    4 warps (8 for 128- and 256-token tiles): tcgen05.ld of the accumulator(s),
//               fused per-channel / per-token scaling, BF16 store of Y; or, for a tile whose
//               K range is cut over several CTAs (split-K or stream-K, see unit_at), a store
//               of the FP32 partial tile into the contributor's workspace slot, after which
//               the last contributor to arrive sums the slots in contributor order and
//               converts.
//   MMA issuers I warps (4 for token tiles up to 64, else 1), each a converged warp whose
//               elected lane issues tcgen05.mma with A = weights in tensor memory (M = 128
//               weight rows) and B = the X tile (N = token_tile rows of X), FP32
//               accumulators in tensor memory.  The weights fill the 128-row side ("swap
//               AB"), so small batches still run full-height MMAs.  A warp needs a few dozen
//               cycles per MMA whatever its size, so narrow token tiles spread the stages
//               over I issuers, each with its own partial accumulator.  BF16 activations use
//               kind::f16; FP8 activations use block-scaled kind::mxf8f6f4 with the E8M0
//               weight scales as scale factors.
//   activation  1 warp (one thread): TMA tiles of X (token_tile rows x 128 bytes per 64-K
//   producer    slab, 128-byte swizzle) into the X ring; for narrow token tiles one 3-D load
//               brings several stages at once.  Indexed MoE (the GATHER instantiations,
//               token tiles up to 64): the whole warp copies the rows that the row index
//               names with cp.async, 16 bytes per lane, into the same swizzled layout.
//   record      1 warp: one bulk copy per stage of the packed weight record (codes, scales
//   producer    and zero points of 128 weight rows x 128 K, see qgemm_internal.h) into the
//               record ring, four lanes issuing four consecutive stages at once.  The ring is
//               deep (up to 16 slots) so that many weight bytes are in flight: small batches
//               are bound by HBM.
//
// Every role walks the CTA's units in the same order (unit_at); the schedule is computed
// once into shared memory after the prologue.
// Stage g of a CTA (counted over all its units) belongs to dequant warpgroup g % W and to
// issuer g % I, and every ring's depth is a multiple of the number of its owners, so each
// slot is always written and read by the same warps.  A waiter that shared a slot with
// another could run two uses ahead, and a one-bit mbarrier parity cannot tell the phase it
// needs from the one before it.
// This follows "Humming wird angekündigt" (vLLM blog, German edition), section "Gemeinsam
// genutzte CUDA-Komponenten" (task scheduling, TMA data movement, dequantization and
// scaling fused into the kernel, tensor-core compute, output stage with fused scaling,
// dense versus MoE scheduling) and section "Leistungsoptimierung basierend auf
// Geräteparametern" (fast MXFP4 -> FP8 conversion for W4A8; Stream-K style split of K).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dequant.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "qgemm_internal.h"

namespace qgemm {

#ifndef QGEMM_DEQ_WGS_NARROW
#define QGEMM_DEQ_WGS_NARROW 4
#endif
#ifndef QGEMM_DEQ_WGS_128
#define QGEMM_DEQ_WGS_128 4
#endif
#ifndef QGEMM_DEQ_WGS_256
#define QGEMM_DEQ_WGS_256 2
#endif
#ifndef QGEMM_EPI_WARPS_256
#define QGEMM_EPI_WARPS_256 16
#endif
#ifndef QGEMM_ISSUERS_NARROW
#define QGEMM_ISSUERS_NARROW 4
#endif
// Warp roles, in this order: the dequant warpgroups, the four epilogue warps, the MMA
// issuers, the activation producer and the record producer.  Groups of four start at a
// multiple of 4, so `warp & 3` is the tensor-memory lane quarter a warp may access.  Every
// SM sub-partition holds a quarter of the warps and of the 64 K registers, so more warps
// leave fewer registers per thread.
// Direct operands (W4A4, and FP8 activations on FP4 operands): no register decode -- the
// MMA reads the weight codes from shared memory, one warpgroup moves the E8M0 scale
// factors into tensor memory, and one issuer runs the stage's MMAs.
template <int BNT, bool D = false, bool A8 = false>
struct Roles {
  // Dequant warpgroups, round-robin over the stages: four up to 128-token tiles, two for
  // 256-token tiles, whose epilogue needs more registers than 27 warps leave (with four it
  // spills and ran up to 15% slower).  The 128-token tile with four instead of two ran up
  // to 8% faster where it is chosen (M = 96 ... 1024) on BF16/FP16 activations and 3-5%
  // slower on FP8 ones (whose decode is a byte shuffle), which keep two.
  static constexpr int kDeqWGs = D ? 1 : BNT <= 64 ? QGEMM_DEQ_WGS_NARROW
                                      : BNT == 128 ? (A8 ? 2 : QGEMM_DEQ_WGS_128)
                                                   : QGEMM_DEQ_WGS_256;
  // An issuing thread needs a few dozen cycles per MMA whatever its size, so narrow token
  // tiles spread the stages over several issuing warps, each with a partial accumulator.
  static constexpr int kIssuers = D ? 1 : BNT <= 64 ? QGEMM_ISSUERS_NARROW : 1;
  // Wide token tiles have one accumulator buffer (or two of 128 columns): several epilogue
  // warps per lane quarter drain it faster, so the MMA waits less for it -- two for
  // 128-token tiles, four for 256-token tiles (64 columns each: the MMA gets the
  // accumulator back after four tensor-memory loads per warp instead of eight, and the
  // kernel needs 72 registers without spilling instead of 96 with).
  static constexpr int kEpiWarps = BNT == 256 ? QGEMM_EPI_WARPS_256 : BNT >= 128 ? 8 : 4;
  static constexpr int kEpiWarp0 = 4 * kDeqWGs;
  static constexpr int kIssuerWarp0 = kEpiWarp0 + kEpiWarps;
  static constexpr int kXProducerWarp = kIssuerWarp0 + kIssuers;
  static constexpr int kRecProducerWarp0 = kXProducerWarp + 1;
  static constexpr int kWarps = kRecProducerWarp0 + 1;
  static constexpr int kThreads = kWarps * 32;
};
constexpr int kMaxExperts = 1024;
// Sleep between polls of a barrier, per role (ns): roles on the critical path poll often,
// the others sleep longer so the dequant warps keep the issue slots.
#ifndef QGEMM_SLEEP_EPI
#define QGEMM_SLEEP_EPI 256
#endif
constexpr uint32_t kSleepDequant = 32, kSleepMma = 32, kSleepProducer = 128,
                   kSleepEpilogue = QGEMM_SLEEP_EPI;
constexpr int kRecTail = kTileN * 4 * 2 + kTileN * 4 / 2;           // largest scales + zeros

constexpr int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }
constexpr int lcm_int(int a, int b) { return a / gcd_int(a, b) * b; }

// A4: W4A4 (MXFP4 activations).  N8: FP8 activations on FP4 operands (A8 as well).
template <int BNT, bool A8, bool A4 = false, bool N8 = false>
struct GemmCfg {
  static_assert(!N8 || A8, "FP4-operand W4A8 has FP8 activations");
  static constexpr bool kDirect = A4 || N8;                      // weights read from smem
  // 32-K chunks per stage: full records, except BF16 x 256 tokens (half records).
  static constexpr int kChunks = (!A8 && !A4 && BNT >= 256) ? 2 : 4;
  static constexpr int kSubStages = 4 / kChunks;                 // stages per record
  // codes + tail; A4: the MMA reads the codes in place, 64-byte-swizzled, so every slot
  // starts on a 512-byte atom; N8: the padded codes (128 rows x 128 bytes, 128-byte
  // swizzle, 1024-byte aligned), the scales in a ring of their own
  static constexpr int kRecSlot = A4 ? 9216 : N8 ? kTileN * 128 : kChunks * kTileN * 16 + kRecTail;
  static constexpr int kTailBytes = N8 ? kTileN * 4 : 0;       // N8: a row's four E8M0 bytes
  // X slabs per stage: 128-byte rows (64 BF16 / 128 FP8 K); A4: one 64-byte row (128 FP4 K)
  static constexpr int kSlabs = (A8 || A4) ? 1 : kChunks / 2;
  static constexpr int kSlabBytes = A4 ? BNT * 64 : BNT * 128;
  static constexpr int kXBytes = kSlabs * kSlabBytes;
  // tensor-memory columns per stage of the A ring: the A operand (BF16 / FP8), or for A4
  // the scale factors (4 for the weights, 4 per 128 tokens for the activations)
  static constexpr int kACols = A4 ? 4 + 4 * ((BNT + 127) / 128) : N8 ? 0 : A8 ? 32 : kChunks * 16;
  static constexpr int kMmaPerStage = A4 ? 2 : A8 ? kChunks : 2 * kChunks;
  static_assert(A4 || A8 || kMmaPerStage % 4 == 0, "BF16 stages issue their MMAs in groups of four");
  static constexpr int kIssuers = Roles<BNT, kDirect, A8>::kIssuers;
  static constexpr int kNumSub = kIssuers;                       // partial accumulators
  static constexpr int kNumAcc = (BNT <= 32 || BNT == 128) ? 2 : 1;  // unit double-buffering
  static constexpr int kAccCols = kNumAcc * kNumSub * BNT;
  // A/X ring depth: what tensor memory holds next to the accumulators (FP8 also needs
  // 4 scale-factor columns per stage and 8 constant ones), capped by shared memory.
  static constexpr int kSfCols = A8 ? 4 : 0;
  static constexpr int kATmemMax = (512 - kAccCols - (A8 ? 8 : 0)) / (kACols + kSfCols);
  static constexpr int kAStagesMax =
      kDirect ? (kATmemMax < 8 ? kATmemMax : 8)
      : A8 ? (BNT >= 128 ? 5 : (kATmemMax < 10 ? kATmemMax : 10))
           : (BNT >= 256 ? 5 : (kATmemMax < 7 ? kATmemMax : 7));
  // Stage g of the CTA goes to dequant warpgroup g % kDeqWGs and to issuer g % kIssuers.
  // A ring slot must always have the same two owners: a waiter that is not the slot's only
  // consumer could run two uses ahead, where a one-bit mbarrier phase parity cannot tell
  // the phase it needs from the one before.  So the depth is a multiple of both counts.
  static constexpr int kDeqWGs = Roles<BNT, kDirect, A8>::kDeqWGs;
  static constexpr int kALcm = lcm_int(kDeqWGs, kIssuers);
  static constexpr int kAStages = kAStagesMax / kALcm * kALcm;
  // X ring: slots of kXChunk stages (one 3-D load per slot for narrow token tiles).
  static constexpr int kXChunk = BNT <= 32 ? 4 : BNT == 64 ? 2 : 1;
  // (N8: only the issuer walks the X ring, which needs no more slots than the record ring
  // keeps stages in flight)
  static constexpr int kXSlots = kXChunk > 1 ? 3 : N8 ? (BNT >= 256 ? 3 : 4) : kAStages;
  // A4: each stage's activation exponents follow the slot's codes, a 16-byte box (four
  // 128-K blocks) per token row
  static constexpr int kXExpBytes = A4 ? BNT * 16 : 0;
  static constexpr int kXSlotBytes = kXChunk * (kXBytes + kXExpBytes);
  static constexpr int kXBoxSlabs = kXChunk * kSlabs;
  static constexpr int kMiscBytes = 64 + 2 * (kMaxExperts + 1) * 4 + BNT * 8;
  static constexpr int kBarBytesPerR = 16, kBarBytesPerA = 16, kBarBytesPerX = 16;
  static constexpr int kFixed = 1024 + kXSlots * (kXSlotBytes + kBarBytesPerX) +
                                kAStages * kBarBytesPerA + kMiscBytes + 64;
  static constexpr int kRMax0 = (227 * 1024 - kFixed) / (kRecSlot + kTailBytes + kBarBytesPerR);
  // record ring: dequant warpgroup g % kDeqWGs (same rule as above)
  static constexpr int kRLcm = kDeqWGs;
  static constexpr int kRMax = kRMax0 / kRLcm * kRLcm;
  static constexpr int kRStages = kRMax < 16 / kRLcm * kRLcm ? kRMax : 16 / kRLcm * kRLcm;
  static constexpr int kACol0 = (kAccCols + 31) / 32 * 32;
  // Block-scale factors (FP8 activations only): per A stage one 4-column slot for the
  // weight-side factors (a row's four E8M0 bytes, one per 32 K, replicated over the four
  // columns of its lane), then 8 columns holding the constant activation-side factor.
  static constexpr int kSfaCol0 = kACol0 + kAStages * kACols;
  static constexpr int kSfbCol0 = (kSfaCol0 + kSfCols * kAStages + 7) / 8 * 8;
  static constexpr int kUsedCols = kSfbCol0 + (A8 ? 8 : 0);
  static constexpr int kTmemCols = kUsedCols <= 32 ? 32 : kUsedCols <= 64 ? 64 :
                                   kUsedCols <= 128 ? 128 : kUsedCols <= 256 ? 256 : 512;
  static_assert(kUsedCols <= 512, "tensor memory budget");
  static_assert(kAStages >= 3 && kRStages >= 4, "pipeline depth");
  static_assert(kAStages % kALcm == 0 && kRStages % kRLcm == 0, "ring slots need fixed owners");
  static constexpr int kBarBytes = kRStages * kBarBytesPerR + kAStages * kBarBytesPerA +
                                   kXSlots * kBarBytesPerX + (2 * kNumAcc + 2) * 8;
  static constexpr int kSmemBytes =
      1024 + kXSlots * kXSlotBytes + kRStages * (kRecSlot + kTailBytes) + kBarBytes + kMiscBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct Unit {
  int nt, mt, expert;
  int kb0, kb1;            // record range [kb0, kb1)
  int64_t row0, row_end;
  // Cut tiles only (ncontrib > 1): arrival counter tile_id; contributor j of the tile
  // keeps its partial sums in workspace slot slot0 + j, j = contrib.
  int tile_id, slot0, contrib, ncontrib;
};

// The schedule of one launch (the same in every CTA; MoE: from the expert offsets) and
// this CTA's part of it, computed once.  Stream-K record counts stay below 2^31 / SMs
// (fewer than SMs tiles of at most 2^16 K blocks), so 32-bit arithmetic is exact.
struct Sched {                 // 7 words: fits misc[8..14] of the kernel's shared memory
  int num_units;           // uniform schedule: units dealt round-robin
  int tiles;               // output tiles
  int sk_tiles;            // > 0: stream-K over tiles [0, sk_tiles), then whole tiles
  uint32_t S;              // stream-K records, sk_tiles * k_blocks
  int lo, hi;              // this CTA's stream-K records [lo, hi)
  int n_sk;                // ... and the pieces (tiles) they fall into
};

static_assert(sizeof(Sched) <= 8 * sizeof(int), "schedule must fit misc[8..15]");

__device__ __forceinline__ Sched make_sched(int num_units, int tiles, int sk_tiles, int k_blocks) {
  Sched sc;
  sc.num_units = num_units;
  sc.tiles = tiles;
  sc.sk_tiles = sk_tiles;
  sc.S = uint32_t(sk_tiles) * uint32_t(k_blocks);
  const uint32_t P = gridDim.x, cta = blockIdx.x;
  sc.lo = int(cta * sc.S / P);
  sc.hi = int((cta + 1) * sc.S / P);
  sc.n_sk = sc.hi > sc.lo ? (sc.hi - 1) / k_blocks - sc.lo / k_blocks + 1 : 0;
  return sc;
}

// Coordinates of output tile `tile`.  Dense: rasterization order, groups of group_m token
// tiles with the token tile changing fastest, so the CTAs running at one time share a few
// weight tiles and the group's activation rows, which stay in L2.  MoE: m-tiles of the
// experts in order, each with its n_tiles weight tiles; `e_hint` is the expert of this
// role's previous tile (tiles only grow along a role's sequence), -1 at the start.
__device__ __forceinline__ void tile_coords(int tile, const GemmArgs& a, int bnt,
                                            const int* prefix, const int* offs, int& e_hint,
                                            Unit& w) {
  const int n_tiles = int(a.L.n_tiles);
  if (a.offsets == nullptr) {
    const int per_group = a.group_m * n_tiles;
    const int first_mt = (tile / per_group) * a.group_m;
    const int gm = min(a.group_m, a.m_tiles - first_mt);
    const int in = tile - (tile / per_group) * per_group;
    w.mt = first_mt + in % gm;
    w.nt = in / gm;
    w.expert = 0;
    w.row0 = int64_t(w.mt) * bnt;
    w.row_end = a.M;
  } else {
    w.nt = tile % n_tiles;
    const int gmt = tile / n_tiles;
    // the largest e < E with prefix[e] <= gmt (empty experts have prefix[e] == prefix[e+1]);
    // binary search above the previous answer (many empty experts may lie in between)
    int lo = e_hint > 0 ? e_hint : 0, hi = a.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= gmt) lo = mid; else hi = mid;
    }
    const int e = lo;
    e_hint = e;
    w.expert = e;
    w.mt = gmt - prefix[e];
    w.row0 = int64_t(offs[e]) + int64_t(w.mt) * bnt;
    w.row_end = offs[e + 1];
  }
}

// The CTA whose stream-K record range holds record x of the S: the largest i with
// floor(i S / P) <= x.
__device__ __forceinline__ int sk_cta_of(uint32_t x, uint32_t S) {
  return int(((x + 1) * gridDim.x - 1) / S);
}

// Unit j (0, 1, ...) of this CTA; false once the CTA has no more.  Every warp role walks
// the same sequence.
//  - uniform: unit u = cta + j P; dense units are (tile, split) pairs, a tile's splits
//    consecutive, splits == 1 meaning whole tiles; MoE units are whole tiles.
//  - stream-K: CTA i first takes records [i S / P, (i + 1) S / P) of the S records of
//    tiles [0, sk_tiles) (pieces of at most two or three tiles), then the whole tiles
//    sk_tiles + i, sk_tiles + i + P, ...  The contributors of a cut tile t are the CTAs
//    first(t) .. last(t) whose ranges meet it; their slots t + first(t) + j never overlap
//    those of another tile, so sk_tiles + P slots hold them all.
__device__ __forceinline__ bool unit_at(int j, const GemmArgs& a, const Sched& sc, int bnt,
                                        const int* prefix, const int* offs, int& e_hint,
                                        Unit& w) {
  const int k_blocks = int(a.L.k_blocks);
  const int P = int(gridDim.x), cta = int(blockIdx.x);
  w.tile_id = 0;
  w.slot0 = 0;
  w.contrib = 0;
  w.ncontrib = 1;
  w.kb0 = 0;
  w.kb1 = k_blocks;
  int tile;
  if (sc.sk_tiles == 0) {
    const int u = cta + j * P;
    if (u >= sc.num_units) return false;
    tile = u;
    if (a.offsets == nullptr && a.splits > 1) {
      const int split = u % a.splits;
      tile = u / a.splits;
      w.kb0 = split * k_blocks / a.splits;
      w.kb1 = (split + 1) * k_blocks / a.splits;
      w.tile_id = tile;
      w.slot0 = tile * a.splits;
      w.contrib = split;
      w.ncontrib = a.splits;
    }
  } else if (j < sc.n_sk) {
    tile = sc.lo / k_blocks + j;
    const int t0 = tile * k_blocks;
    w.kb0 = j == 0 ? sc.lo - t0 : 0;
    w.kb1 = min(sc.hi, t0 + k_blocks) - t0;
    const int first = sk_cta_of(uint32_t(t0), sc.S);
    const int last = sk_cta_of(uint32_t(t0 + k_blocks - 1), sc.S);
    if (last > first) {
      w.tile_id = tile;
      if (sc.S >= uint32_t(P)) {
        // every CTA holds a record, so the tile's contributors are CTAs first..last
        w.slot0 = tile + first;
        w.contrib = cta - first;
        w.ncontrib = last - first + 1;
      } else {
        // fewer records than CTAs: each CTA holds at most one, and some none, so the
        // contributors are the owners of the tile's k_blocks records, in record order
        // (slot = the record's index, below S)
        w.slot0 = t0;
        w.contrib = sc.lo - t0;
        w.ncontrib = k_blocks;
      }
    }
  } else {
    tile = sc.sk_tiles + cta + (j - sc.n_sk) * P;
    if (tile >= sc.tiles) return false;
  }
  tile_coords(tile, a, bnt, prefix, offs, e_hint, w);
  return true;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// One arrival per warp once every lane got here (barriers of warp roles count warps, not
// threads: 128 per-thread arrivals would serialise on the barrier's shared-memory word).
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(bar);
}

// Release a shared-memory slot that this warp read with ordinary loads to a producer that
// refills it with bulk copies: every lane orders its reads before the copies (which write
// through the async proxy) with a proxy fence, then one arrival is made.  Without the
// fence the refill could overwrite the slot before all reads of it were performed, which
// showed as a lane quarter of a tile decoded from the next record.
__device__ __forceinline__ void release_to_async(uint64_t* bar, int lane) {
  ptx::fence_proxy_async_smem();
  warp_arrive(bar, lane);
}

// Position in a ring of `n` slots: slot index and the parity of its current use.
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) { slot = 0; phase ^= 1u; }
  }
};

// Decode modes: the kernel is compiled per weight format so that the decode loop holds
// only the code it runs.  "G1": one scale (and zero point) per row per record, i.e. a
// group of 128 K or longer, so they are read once per record.
enum DecodeMode : int {
  DM_INT4_ZP_G1 = 0, DM_INT4_SYM_G1 = 1, DM_INT4_ANY = 2, DM_MXFP4 = 3, DM_MXINT4 = 4, DM_NVFP4 = 5,
  DM_W4A4 = 6,                 // MXFP4 x MXFP4: no decode, the MMA reads the codes
  DM_W4A8N = 7,                // MXFP4 x FP8 on FP4 operands: no decode either
  DM_MXFP4_F16 = 8,            // MXFP4 x BF16 activations on FP16 operands (narrow tiles)
  DM_NVFP4_F16 = 9             // NVFP4, likewise
};

// INT4 with BF16 scales (every group size) and MXFP4 in small calls: FP16 tensor-core
// operands, see f16_operands() and mx_f16_capable().
template <bool A8, int DM>
constexpr bool kF16Operands =
    !A8 && (DM == DM_INT4_ZP_G1 || DM == DM_INT4_SYM_G1 || DM == DM_INT4_ANY ||
            DM == DM_MXFP4_F16 || DM == DM_NVFP4_F16);

// Decode two 32-K chunks of weight row r into 32 registers of 16-bit pairs (pair order):
// FP16 for INT4 with BF16 scales (the scale times w_pre = 2^k), BF16 for the other formats.
// The codes come from slot chunks `slot0`, `slot0 + 1` of the staged record; their scales
// and zero points are the record's entries for record chunks `rchunk0`, `rchunk0 + 1`.
template <int DM>
__device__ __forceinline__ void decode_two_chunks_a16(const uint8_t* rec, int tail, int slot0,
                                                      int rchunk0, int r, int has_zp, int G,
                                                      int zoff, float w_pre, uint32_t (&regs)[32]) {
  if constexpr (DM == DM_INT4_ZP_G1 || DM == DM_INT4_SYM_G1) {
    const uint32_t s = reinterpret_cast<const uint16_t*>(rec + tail)[r];
    uint32_t z = 8;
    if constexpr (DM == DM_INT4_ZP_G1) z = (rec[tail + zoff + (r >> 1)] >> (4 * (r & 1))) & 0xFu;
    const uint32_t zz = (0x6400u | z) * 0x00010001u, zz64 = (0x5400u | (z << 4)) * 0x00010001u;
    const uint32_t s2 = scale_f16x2(s, w_pre);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 q = *reinterpret_cast<const uint4*>(rec + (slot0 + c) * (kTileN * 16) + r * 16);
      const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) decode_int4_word_f16(wd[j], zz, zz64, s2, &regs[16 * c + 4 * j]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 q = *reinterpret_cast<const uint4*>(rec + (slot0 + c) * (kTileN * 16) + r * 16);
      const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
      if constexpr (DM == DM_MXFP4) {
        const uint32_t E = rec[tail + r * 4 + rchunk0 + c];   // one E8M0 per 32 K
        uint32_t sa, sb;
        bool big;
        mxfp4_factors(E, sa, sb, big);
        const bool two = __any_sync(0xffffffffu, big);
#pragma unroll
        for (int j = 0; j < 4; ++j) decode_mxfp4_word_nat(wd[j], sa, sb, two, &regs[16 * c + 4 * j]);
      } else if constexpr (DM == DM_MXFP4_F16) {
        const uint32_t f2 = e8m0_f16x2(rec[tail + r * 4 + rchunk0 + c], w_pre);
#pragma unroll
        for (int j = 0; j < 4; ++j) decode_mxfp4_word_f16(wd[j], f2, &regs[16 * c + 4 * j]);
      } else if constexpr (DM == DM_MXINT4) {
        const uint32_t s2 = e8m0_bf16x2(rec[tail + r * 4 + rchunk0 + c]);   // one E8M0 per 32 K
#pragma unroll
        for (int j = 0; j < 4; ++j) decode_int4_word(wd[j], 0x43084308u, s2, &regs[16 * c + 4 * j]);
      } else if constexpr (DM == DM_NVFP4) {
        // one E4M3 scale per 16 K: words 0, 1 of the chunk take the first, words 2, 3 the second
        const uint32_t sp = reinterpret_cast<const uint16_t*>(rec + tail)[r * 4 + rchunk0 + c];
        const uint32_t s0 = e4m3_bf16x2_p118(sp & 0xFFu), s1 = e4m3_bf16x2_p118(sp >> 8);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          decode_mxfp4_word_nat(wd[j], j < 2 ? s0 : s1, 0u, false, &regs[16 * c + 4 * j]);
      } else if constexpr (DM == DM_NVFP4_F16) {
        // the chunk's two E4M3 scales (16 K each) -> f16x2, times 16 (exact: e2m1 x E4M3 x 16
        // stays within FP16's normal range), each broadcast to both halves
        const uint32_t sp = reinterpret_cast<const uint16_t*>(rec + tail)[r * 4 + rchunk0 + c];
        const uint32_t ss = ptx::f16x2_mul(ptx::cvt_f16x2_e4m3x2(sp), 0x4C004C00u);
        const uint32_t s0 = ptx::prmt(ss, ss, 0x1010u), s1 = ptx::prmt(ss, ss, 0x3232u);
#pragma unroll
        for (int j = 0; j < 4; ++j) decode_mxfp4_word_f16(wd[j], j < 2 ? s0 : s1, &regs[16 * c + 4 * j]);
      } else {
        const int ent = r * G + ((rchunk0 + c) * G) / 4;      // scale entry of this chunk
        const uint32_t s = reinterpret_cast<const uint16_t*>(rec + tail)[ent];
        uint32_t z = 8;
        if (has_zp) z = (rec[tail + zoff + (ent >> 1)] >> (4 * (ent & 1))) & 0xFu;
        const uint32_t zz = (0x6400u | z) * 0x00010001u, zz64 = (0x5400u | (z << 4)) * 0x00010001u;
        const uint32_t s2 = scale_f16x2(s, w_pre);
#pragma unroll
        for (int j = 0; j < 4; ++j) decode_int4_word_f16(wd[j], zz, zz64, s2, &regs[16 * c + 4 * j]);
      }
    }
  }
}

// One gathered row of an activation slot: 16 bytes at src + s * 128 into dst + s * SLAB for
// the S slabs s (src and dst already include the lane's piece).
template <int S, int SLAB, int I = 0>
__device__ __forceinline__ void gather_row(uint32_t dst, const uint8_t* src, uint64_t pol) {
  if constexpr (I < S) {
    ptx::cp_async_16_at<I * SLAB, I * 128>(dst, src, pol);
    gather_row<S, SLAB, I + 1>(dst, src, pol);
  }
}

template <int BNT, bool A8, int DM, bool GATHER>
__global__ void __launch_bounds__(Roles<BNT, DM == DM_W4A4 || DM == DM_W4A8N, A8>::kThreads, 1)
qgemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ GemmArgs a) {
  static_assert(!GATHER || BNT <= 64, "gathered tiles exist for token tiles up to 64");
  constexpr bool A4 = DM == DM_W4A4;
  constexpr bool N8 = DM == DM_W4A8N;
  constexpr bool kDirect = A4 || N8;       // the MMA reads the weight codes from shared memory
  static_assert(!A4 || (!A8 && !GATHER), "W4A4: its own activation format, TMA loads only");
  static_assert(!N8 || A8, "FP4-operand W4A8: FP8 activations");
  constexpr bool F16 = kF16Operands<A8, DM>;
  // per-token (per-row) output scale: FP8's token scale, or the FP16 copy's row scale
  constexpr bool kTokScale = A8 || F16;
  using C = GemmCfg<BNT, A8, A4, N8>;
  using RO = Roles<BNT, kDirect, A8>;
  constexpr int kEpiWarp0 = RO::kEpiWarp0;
  constexpr int kDeqWGs = RO::kDeqWGs;
  constexpr int kXProducerWarp = RO::kXProducerWarp;
  constexpr int SA = C::kAStages;
  constexpr int SR = C::kRStages;
  constexpr int SX = C::kXSlots;
  constexpr int XQ = C::kXChunk;
  constexpr int CH = C::kChunks;
  constexpr int kSub = C::kSubStages;
  constexpr int kTail = CH * kTileN * 16;                // scales + zeros inside a slot
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_x = smem;                                   // [SX][kXSlotBytes], 1024-aligned
  uint8_t* s_rec = s_x + SX * C::kXSlotBytes;            // [SR][kRecSlot]
  uint8_t* s_tail = s_rec + SR * C::kRecSlot;            // N8: [SR][kTailBytes] scales
  uint64_t* rfull = reinterpret_cast<uint64_t*>(s_tail + SR * C::kTailBytes);
  uint64_t* rempty = rfull + SR;
  uint64_t* xfull = rempty + SR;
  uint64_t* xempty = xfull + SX;
  uint64_t* afull = xempty + SX;
  uint64_t* aempty = afull + SA;
  uint64_t* accfull = aempty + SA;
  uint64_t* accempty = accfull + C::kNumAcc;
  uint64_t* drain = accempty + C::kNumAcc;
  uint64_t* epibar = drain + 1;                          // epilogue rendezvous (split-K)
  // misc: [0] tmem [1] abort [2] ok [3] units [4] last arriver [8..14] schedule (Sched)
  int* misc = reinterpret_cast<int*>(epibar + 1);
                                                         // [8..14] schedule (Sched)
  int* prefix = misc + 16;                               // MoE: m-tiles before expert e
  int* offs = prefix + (kMaxExperts + 1);                // MoE: row offsets
  int* idx_s = offs + (kMaxExperts + 1);                 // indexed MoE: X row offsets (int64)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Layout& L = a.L;

  // ------------------------------------------------------------------ prologue
  // The header loads are issued first and checked after the barrier set-up, and tensor
  // memory is allocated at the same time, so that their latencies overlap.
  if (threadIdx.x == 0) {
    const PackedHeader* h = reinterpret_cast<const PackedHeader*>(a.packed);
    const PackedHeader hd = *h;
    const PackedHeader* hl = reinterpret_cast<const PackedHeader*>(
        a.packed + int64_t(a.offsets != nullptr && a.E > 1 ? a.E - 1 : 0) * a.expert_stride);
    const uint32_t hl_magic = hl->magic;
    const int64_t hl_N = hl->N, hl_K = hl->K;
    const int32_t hl_afmt = hl->afmt;
    misc[1] = 0;
    for (int s = 0; s < SR; ++s) {
      ptx::mbar_init(&rfull[s], 1);
      ptx::mbar_init(&rempty[s], kDirect ? 1 : 4);   // per dequant warp; direct: the MMAs' commit
    }
    for (int s = 0; s < SX; ++s) {
      ptx::mbar_init(&xfull[s], GATHER ? 32 : 1);   // gathered slots: one arrival per lane
      ptx::mbar_init(&xempty[s], C::kIssuers);
    }
    for (int s = 0; s < SA; ++s) {
      ptx::mbar_init(&afull[s], 4);
      ptx::mbar_init(&aempty[s], 1);
    }
    for (int i = 0; i < C::kNumAcc; ++i) {
      ptx::mbar_init(&accfull[i], C::kIssuers);
      ptx::mbar_init(&accempty[i], RO::kEpiWarps);  // one arrival per epilogue warp
    }
    ptx::mbar_init(drain, C::kIssuers);
    ptx::mbar_init(epibar, RO::kEpiWarps);
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    bool ok = hd.magic == kPackedMagic && hd.version == kPackedVersion && hd.wfmt == L.wfmt &&
              hd.group == L.group && hd.has_zp == L.has_zp && hd.afmt == L.afmt &&
              hd.N == L.N && hd.K == L.K && hd.total_bytes == L.total_bytes;
    // MoE: the last expert's header as well
    ok = ok && hl_magic == kPackedMagic && hl_N == L.N && hl_K == L.K && hl_afmt == L.afmt;
    if (!ok) atomicCAS(a.status, 0, kStatusBadPacked);
    // the gathering variant runs exactly the indexed calls
    if (ok && (a.row_index != nullptr) != GATHER) {
      atomicCAS(a.status, 0, kStatusBadValue);
      ok = false;
    }
    misc[2] = ok ? 1 : 0;
  }
  if (warp == kEpiWarp0) {
    ptx::tmem_alloc(reinterpret_cast<uint32_t*>(&misc[0]), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if constexpr (!GATHER)
    if (warp == kXProducerWarp && lane == 0) ptx::prefetch_tmap(&tmap_x);
  if constexpr (N8)
    if (warp == RO::kRecProducerWarp0 && lane == 0) ptx::prefetch_tmap(&a.tmap_w);
  int num_units = a.num_units;
  if (a.offsets != nullptr && warp == 0) {
    // MoE schedule: m-tiles per expert and their exclusive prefix (one warp).  All offsets
    // are loaded first (independent loads, one memory latency), then scanned from shared
    // memory.
    for (int base = 0; base <= a.E; base += 32 * 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = base + j * 32 + lane;
        v[j] = e <= a.E ? __ldg(a.offsets + e) : 0;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = base + j * 32 + lane;
        if (e <= a.E) offs[e] = v[j];
      }
    }
    __syncwarp();
    int carry = 0;
    bool bad = false;
    for (int base = 0; base <= a.E; base += 32) {
      const int e = base + lane;
      int t = 0;
      if (e < a.E) {
        const int o = offs[e], o1 = offs[e + 1];
        if (o1 < o || o < 0 || o1 > a.M) bad = true;
        t = (o1 > o) ? (o1 - o + BNT - 1) / BNT : 0;
      }
      int incl = t;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      if (e <= a.E) prefix[e] = carry + incl - t;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      misc[3] = bad ? 0 : carry;
      if (bad) atomicCAS(a.status, 0, kStatusBadValue);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  int tiles = a.m_tiles * int(L.n_tiles), sk_tiles = a.sk_tiles;
  if (a.offsets != nullptr) {
    // MoE: the tile count is known only now.  With a workspace, stream-K over the leftover
    // tiles when every CTA's share is at least 16 K blocks (shorter pieces cost more in
    // partial sums than the better balance saves).
    num_units = tiles = misc[3] * int(L.n_tiles);
    const int P = int(gridDim.x);
    const int left = tiles < P ? tiles : tiles % P;
    sk_tiles = (a.ws != nullptr && int64_t(left) * L.k_blocks >= 16 * int64_t(P)) ? left : 0;
  }
  const uint32_t tbase = static_cast<uint32_t>(misc[0]);
  if (!misc[2] || (sk_tiles == 0 && int(blockIdx.x) >= num_units)) {   // nothing to do
    if (warp == kEpiWarp0) ptx::tmem_dealloc(tbase, C::kTmemCols);
    return;
  }
  // The schedule lives in shared memory (written once, read once per unit) rather than in
  // registers of every role.
  Sched* sched = reinterpret_cast<Sched*>(misc + 8);
  if (threadIdx.x == 0) *sched = make_sched(num_units, tiles, sk_tiles, int(L.k_blocks));
  volatile int* abort_flag = &misc[1];
  const uint64_t T = a.timeout_ns;

  if (A8 && warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {    // first lane quarter set
    // Activation-side block scale: a constant 2^6 (E8M0 133) that returns the factor 2^-6
    // of the e2m1 -> e4m3 byte shuffle; on FP4 operands 1 (E8M0 127).  Filled over every
    // lane of its columns.
    const uint32_t tl = tbase + (uint32_t((warp & 3) * 32) << 16);
    constexpr uint32_t sfb = N8 ? 0x7F7F7F7Fu : 0x85858585u;
    ptx::tmem_st4(tl + C::kSfbCol0, sfb, sfb, sfb, sfb);
    ptx::tmem_st4(tl + C::kSfbCol0 + 4, sfb, sfb, sfb, sfb);
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const Sched& sc = *sched;

  if (warp >= RO::kRecProducerWarp0) {
    // ---------------------------------------------------------------- record producer
    // One warp walks the stages in order, kCopyLanes consecutive stages of a unit at a
    // time, one lane per stage: the lanes issue their bulk copies together.  Issuing a copy
    // keeps its thread busy for a few hundred cycles, and copies issued by different lanes
    // overlap, so one SM streams about twice as many bytes per cycle as from a single
    // thread.  The warp stays converged from one group to the next, so the waits on any
    // one slot follow the stage order, whichever lane makes them.
    // (wide token tiles: one lane; four measured 2% slower at 7168 x 2048, M = 8192)
    constexpr int kCopyLanes = BNT >= 128 ? 1 : 4;
    constexpr uint32_t kLaneMask = (1u << kCopyLanes) - 1u;
    if (lane < kCopyLanes) {
    const uint64_t pol_w = a.m_tiles <= 1 ? ptx::policy_evict_first() : ptx::policy_evict_normal();
    const uint32_t rec_bytes = uint32_t(L.record_bytes);
    const uint32_t tail_bytes = rec_bytes - uint32_t(kCodeBytes);     // scales + zeros
    // (N8: the tensor copy counts the packed bytes it reads, not the padded ones it writes)
    const uint32_t stage_tx = N8 ? uint32_t(kCodeBytes + C::kTailBytes)
                              : CH == 4 ? rec_bytes : uint32_t(kCodeBytes / 2) + tail_bytes;
    uint32_t g0 = 0;                    // CTA stage counter at the unit start
    uint32_t fail_g = 0, fail_iss = 0;  // on a failed wait: the group's first stage and its issued lanes
    bool alive = true;
    Unit w;
    int e_hint = -1;
    for (int uj = 0; alive && unit_at(uj, a, sc, BNT, prefix, offs, e_hint, w); ++uj) {
      const uint8_t* rec0 = a.packed + int64_t(w.expert) * a.expert_stride + kHeaderBytes +
                            (int64_t(w.nt) * L.k_blocks + w.kb0) * int64_t(rec_bytes);
      const int nst = (w.kb1 - w.kb0) * kSub;
      for (int i0 = 0; i0 < nst; i0 += kCopyLanes) {
        const int i = i0 + lane;                        // this lane's stage of the unit
        const uint32_t g = g0 + uint32_t(i);
        const int slot = int(g % uint32_t(SR));
        const uint32_t ph = (g / uint32_t(SR)) & 1u;
        bool ok = true, issued = false;
        if (i < nst) {
          ok = ptx::mbar_wait(&rempty[slot], ph ^ 1u, abort_flag, T, kSleepProducer);
          if (ok) {
            const uint8_t* rec = rec0 + int64_t(i / kSub) * rec_bytes;
            uint8_t* sr = s_rec + slot * C::kRecSlot;
            ptx::mbar_arrive_expect_tx(&rfull[slot], stage_tx);
            if constexpr (N8) {
              // the codes through the tensor map, which writes them as padded 128-byte rows;
              // the scales as plain bytes into the slot's tail
              const int32_t ridx = int32_t(int64_t(w.nt) * L.k_blocks + w.kb0 + i);
              ptx::tma_load_4d(sr, &a.tmap_w, 0, 0, ridx, w.expert, &rfull[slot], pol_w);
              ptx::bulk_g2s(s_tail + slot * C::kTailBytes, rec + kCodeBytes, C::kTailBytes,
                            &rfull[slot], pol_w);
            } else if (CH == 4) {
              ptx::bulk_g2s(sr, rec, rec_bytes, &rfull[slot], pol_w);
            } else {
              // half record: codes of record chunks 2h, 2h+1, then the scales and zeros
              const int h = i % kSub;
              ptx::bulk_g2s(sr, rec + h * (kCodeBytes / 2), kCodeBytes / 2, &rfull[slot], pol_w);
              ptx::bulk_g2s(sr + kTail, rec + kCodeBytes, tail_bytes, &rfull[slot], pol_w);
            }
            issued = true;
          }
        }
        if (!__all_sync(kLaneMask, ok)) {
          alive = false;
          fail_g = g0 + uint32_t(i0);
          fail_iss = __ballot_sync(kLaneMask, issued);
          break;
        }
      }
      g0 += uint32_t(nst);
    }
    if (!alive && lane == 0) {
      // Let every copy the warp issued land first.  Every stage before fail_g was issued,
      // and of the group at fail_g the lanes in fail_iss; each slot's last fill is waited
      // for (an earlier fill of the slot was consumed, so it has landed).
      volatile int no_abort = 0;
      const uint32_t lo = fail_g > uint32_t(SR) ? fail_g - uint32_t(SR) : 0u;
      for (uint32_t g = lo; g < fail_g + uint32_t(kCopyLanes); ++g) {
        const bool in_group = g >= fail_g;
        if (in_group && !((fail_iss >> (g - fail_g)) & 1u)) continue;       // not issued
        if (!in_group && g + uint32_t(SR) >= fail_g && g + uint32_t(SR) < fail_g + uint32_t(kCopyLanes) &&
            ((fail_iss >> (g + uint32_t(SR) - fail_g)) & 1u))
          continue;                                                         // refilled later
        ptx::mbar_wait(&rfull[g % uint32_t(SR)], (g / uint32_t(SR)) & 1u, &no_abort, 200000000ull);
      }
    }
    }
  } else if (warp == kXProducerWarp) {
    // ---------------------------------------------------------------- activation producer
    // FP16 operands: the activations come from the pre-pass launched just before
    if constexpr (F16) ptx::grid_dependency_wait();
    if constexpr (A4)
      if (lane == 0) ptx::prefetch_tmap(&a.tmap_e);
    if constexpr (GATHER) {
      // Gathered (indexed MoE) tiles: the warp copies each unit's rows out of X in token
      // order, 16 bytes per lane and copy (cp.async), straight into the 128-byte-swizzled
      // layout that the MMA reads (16-byte piece j of tile row i sits at piece j xor (i mod 8)
      // of the row's 128 bytes).  The eight lanes of a group cover one 128-byte line, so each
      // instruction reads four whole lines, and a lane keeps its row's source offset over
      // the slabs.  Rows past the end of the expert's block are not copied: their
      // accumulator columns are never stored, and MMA column n reads activation row n only.
      // Each lane hands its copies of a slot to the slot's barrier (32 arrivals,
      // each made by the hardware once that lane's copies have landed), so the warp never
      // waits for its own copies and runs up to the ring's depth ahead.  The copies land in
      // the generic proxy: the MMA issuers fence them for the tensor cores after their wait.
      // Negative indices and columns past K are zero-filled; an index past the end of X
      // sets the error status and reads zeros.
      constexpr int kEsz = A8 ? 1 : 2;
      const uint64_t pol_x = ptx::policy_evict_last();
      int64_t* xoff_s = reinterpret_cast<int64_t*>(idx_s);
      const int grp = lane >> 3, ch = lane & 7;
      Ring rx;
      bool alive = true;
      Unit w;
      int e_hint = -1;
      for (int uj = 0; alive && unit_at(uj, a, sc, BNT, prefix, offs, e_hint, w); ++uj) {
        __syncwarp();                     // every lane is done with the previous unit's rows
        const int nrows = w.row_end - w.row0 < BNT ? int(w.row_end - w.row0) : BNT;
        for (int i = lane; i < nrows; i += 32) {
          const int32_t t = __ldg(a.row_index + w.row0 + i);
          if (t >= a.x_rows) atomicCAS(a.status, 0, kStatusBadValue);
          xoff_s[i] = t >= 0 && t < a.x_rows ? int64_t(t) * a.ldx_bytes : -1;
        }
        __syncwarp();
        const int nst = (w.kb1 - w.kb0) * kSub;
        for (int i0 = 0; i0 < nst; i0 += XQ) {
          if (!warp_all(ptx::mbar_wait(&xempty[rx.slot], rx.phase ^ 1u, abort_flag, T, kSleepProducer))) { alive = false; break; }
          const uint32_t sx = ptx::smem_u32(s_x + rx.slot * C::kXSlotBytes);
          // first column (elements) of this lane's piece in the slot's first slab, and the
          // number of the slot's slabs in which that piece lies before K (K is a multiple of
          // 32, so a piece is wholly inside K or wholly past it)
          const int64_t c0 = int64_t(w.kb0) * kStageK + i0 * (kStageK / kSub) + ch * (16 / kEsz);
          const int64_t left = (L.K - c0 + 128 / kEsz - 1) / (128 / kEsz);
          const int n_in = left <= 0 ? 0 : left < C::kXBoxSlabs ? int(left) : C::kXBoxSlabs;
          const uint8_t* xk = a.x + c0 * kEsz;
#pragma unroll 2
          for (int i = grp; i < nrows; i += 4) {
            const int64_t off = xoff_s[i];
            const uint32_t dst = sx + uint32_t(i * 128 + ((ch ^ (i & 7)) << 4));
            if (off >= 0 && n_in == C::kXBoxSlabs) {
              gather_row<C::kXBoxSlabs, C::kSlabBytes>(dst, xk + off, pol_x);
            } else {
#pragma unroll
              for (int sl = 0; sl < C::kXBoxSlabs; ++sl) {
                const bool in = off >= 0 && sl < n_in;
                ptx::cp_async_16(dst + sl * C::kSlabBytes, in ? xk + off + sl * 128 : a.x,
                                 in ? 16u : 0u, pol_x);
              }
            }
          }
          ptx::cp_async_arrive_noinc(&xfull[rx.slot]);
          rx.next(SX);
        }
      }
      ptx::cp_async_wait_all();           // nothing of this warp is left in flight at exit
    } else if (lane == 0) {
      // every X tile is read by all weight tiles of its group: keep it in L2
      const uint64_t pol_x = ptx::policy_evict_last();
      Ring rx;
      uint32_t pending = 0, pending_parity = 0;
      bool alive = true;
      Unit w;
      int e_hint = -1;
      for (int uj = 0; alive && unit_at(uj, a, sc, BNT, prefix, offs, e_hint, w); ++uj) {
        const int32_t row0 = int32_t(w.row0);
        const int nst = (w.kb1 - w.kb0) * kSub;
        for (int i0 = 0; i0 < nst; i0 += XQ) {
          if (!ptx::mbar_wait(&xempty[rx.slot], rx.phase ^ 1u, abort_flag, T, kSleepProducer)) { alive = false; break; }
          if (a.debug_skip_first_x && uj == 0 && i0 == 0) {   // test aid: issue nothing
            rx.next(SX);
            continue;
          }
          uint8_t* sx = s_x + rx.slot * C::kXSlotBytes;
          // K offset (elements) of the chunk's first stage: records kb0.., sub-stage h
          const int k0 = w.kb0 * kStageK + i0 * (kStageK / kSub);
          ptx::mbar_arrive_expect_tx(&xfull[rx.slot], uint32_t(C::kXSlotBytes));
          if constexpr (A4) {
            // the exponents of each stage: x = 16-byte group of its 128-K block
#pragma unroll 1
            for (int sl = 0; sl < C::kXBoxSlabs; ++sl) {
              const int kb = k0 / kStageK + sl;
              ptx::tma_load_2d(sx + C::kXChunk * C::kXBytes + sl * C::kXExpBytes, &a.tmap_e,
                               (kb >> 2) * 16, row0, &xfull[rx.slot], pol_x);
            }
          }
          if (a.x_3d) {
            // box {slab, token_tile rows, kXBoxSlabs slabs}; slab index = K / slab width
            ptx::tma_load_3d(sx, &tmap_x, 0, row0, k0 / (A8 ? 128 : 64), &xfull[rx.slot], pol_x);
          } else {
#pragma unroll 1
            for (int sl = 0; sl < C::kXBoxSlabs; ++sl)   // (A4: the map counts bytes of codes)
              ptx::tma_load_2d(sx + sl * C::kSlabBytes, &tmap_x,
                               A4 ? k0 / 2 + sl * 64 : k0 + sl * (A8 ? 128 : 64), row0,
                               &xfull[rx.slot], pol_x);
          }
          pending |= 1u << rx.slot;
          pending_parity = (pending_parity & ~(1u << rx.slot)) | (rx.phase << rx.slot);
          rx.next(SX);
        }
      }
      if (!alive) {
        volatile int no_abort = 0;
        for (int s = 0; s < SX; ++s)
          if (pending & (1u << s))
            ptx::mbar_wait(&xfull[s], (pending_parity >> s) & 1u, &no_abort, 200000000ull);
      }
    }
  } else if (warp >= RO::kIssuerWarp0 && warp < kXProducerWarp) {
    // ---------------------------------------------------------------- MMA issuers
    // Issuer j takes the stages g of this CTA with g % kIssuers == j and accumulates into
    // partial accumulator j.  The whole warp runs the loop and one elected lane issues: a
    // converged warp issues tcgen05 instructions faster than a lone diverged lane.
    const int issuer = warp - RO::kIssuerWarp0;
    Ring rx;
    int ui = 0;
    uint32_t g0 = 0;                      // CTA stage counter at the unit start
    bool alive = true;
    const uint64_t desc0 = A4 ? ptx::desc_kmajor_sw64(ptx::smem_u32(s_x))
                              : ptx::desc_kmajor_sw128(ptx::smem_u32(s_x));
    Unit w;
    int e_hint = -1;
    for (int uj = 0; alive && unit_at(uj, a, sc, BNT, prefix, offs, e_hint, w); ++uj, ++ui) {
      const int acc = ui % C::kNumAcc;
      const uint32_t acc_par = uint32_t((ui / C::kNumAcc) & 1);
      if (!warp_all(ptx::mbar_wait(&accempty[acc], acc_par ^ 1u, abort_flag, T, kSleepMma))) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tbase + uint32_t((acc * C::kNumSub + issuer) * BNT);
      const int nst = (w.kb1 - w.kb0) * kSub;
      uint32_t first = 1;                 // this issuer's first MMA of the unit overwrites
      for (int x0 = 0; x0 < nst && alive; x0 += XQ) {
        // Every issuer waits for every X slot, even one without a stage of its own: its
        // release of the slot below must count towards this fill of the slot, not the next.
        if (!warp_all(ptx::mbar_wait(&xfull[rx.slot], rx.phase, abort_flag, T, kSleepMma))) { alive = false; break; }
        // gathered slots were written by cp.async (generic proxy): order them before the
        // tensor cores read them
        if constexpr (GATHER) ptx::fence_proxy_async_smem();
        const int x1 = x0 + XQ < nst ? x0 + XQ : nst;
        // this issuer's stages in [x0, x1): CTA stage g0 + i with (g0 + i) % kIssuers == issuer
        const uint32_t gx = g0 + uint32_t(x0);
        int i = x0 + int((uint32_t(issuer) + uint32_t(C::kIssuers) - gx % uint32_t(C::kIssuers)) %
                         uint32_t(C::kIssuers));
        for (; i < x1; i += C::kIssuers) {
          const uint32_t g = g0 + uint32_t(i);
          const int xj = i - x0;          // stage inside the X slot
          Ring cur;
          cur.slot = int(g % uint32_t(SA));
          cur.phase = (g / uint32_t(SA)) & 1u;
          if (!warp_all(ptx::mbar_wait(&afull[cur.slot], cur.phase, abort_flag, T, kSleepMma))) { alive = false; break; }
          ptx::tc_fence_after();
          const uint64_t bdesc = desc0 + uint64_t((rx.slot * C::kXSlotBytes + xj * C::kXBytes) >> 4);
          const uint32_t a_tmem = tbase + uint32_t(C::kACol0 + cur.slot * C::kACols);
          if constexpr (A4) {
            // A is the stage's record in shared memory; the A "slot" holds its scale factors
            const int rs = int(g % uint32_t(SR));
            if (!warp_all(ptx::mbar_wait(&rfull[rs], (g / uint32_t(SR)) & 1u, abort_flag, T, kSleepMma))) { alive = false; break; }
            ptx::tc_fence_after();
            const uint64_t adesc = ptx::desc_kmajor_sw64(ptx::smem_u32(s_rec + rs * C::kRecSlot));
#pragma unroll
            for (int q = 0; q < 2; ++q)   // two 64-K steps: 32 bytes into the swizzled rows
              ptx::mma_mxf4_ss_elect(d_tmem, adesc + uint64_t(q * 2), bdesc + uint64_t(q * 2),
                                     ptx::idesc_mxf4(128, BNT, 2 * q, 2 * q), a_tmem, a_tmem + 4u,
                                     q > 0 ? 1u : (first ^ 1u));
            first = 0;
            ptx::mma_commit_elect(&aempty[cur.slot]);   // frees the stage's scale factors
            ptx::mma_commit_elect(&rempty[rs]);         // ... and its record
            continue;
          }
          if constexpr (N8) {
            // A is the stage's padded e2m1 codes in shared memory, B the FP8 tile: four
            // K = 32 MMAs, each with its byte of the rows' E8M0 scale words
            const int rs = int(g % uint32_t(SR));
            if (!warp_all(ptx::mbar_wait(&rfull[rs], (g / uint32_t(SR)) & 1u, abort_flag, T, kSleepMma))) { alive = false; break; }
            ptx::tc_fence_after();
            const uint64_t adesc = ptx::desc_kmajor_sw128(ptx::smem_u32(s_rec + rs * C::kRecSlot));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)   // 32 bytes (32 K) into the 128-byte rows
              ptx::mma_mxf8f6f4_ss_elect(d_tmem, adesc + uint64_t(kk * 2), bdesc + uint64_t(kk * 2),
                                         ptx::idesc_mxf8_e2m1_e4m3(128, BNT, kk, 0),
                                         tbase + uint32_t(C::kSfaCol0 + 4 * cur.slot),
                                         tbase + uint32_t(C::kSfbCol0),
                                         kk > 0 ? 1u : (first ^ 1u));
            first = 0;
            ptx::mma_commit_elect(&aempty[cur.slot]);   // frees the stage's scale factors
            ptx::mma_commit_elect(&rempty[rs]);         // ... and its record
            continue;
          }
          if constexpr (A8) {
#pragma unroll
            for (int kk = 0; kk < C::kMmaPerStage; ++kk) {
              const uint32_t accum = kk > 0 ? 1u : (first ^ 1u);
              ptx::mma_mxf8f6f4_ts_elect(d_tmem, a_tmem + kk * 8, bdesc + uint64_t(kk * 2),
                                         ptx::idesc_mxf8_e4m3(128, BNT, kk, 0),
                                         tbase + uint32_t(C::kSfaCol0 + 4 * cur.slot),
                                         tbase + uint32_t(C::kSfbCol0), accum);
            }
          } else {
            // one 128-byte slab (64 K) per group of four: 32-byte K steps inside its swizzled
            // rows, the four MMAs issued under one election
#pragma unroll
            for (int q = 0; q < C::kMmaPerStage / 4; ++q) {
              const uint64_t b = bdesc + uint64_t((q * C::kSlabBytes) >> 4);
              const uint32_t a = a_tmem + uint32_t(q * 32);
              ptx::mma4_f16_ts_elect(d_tmem, a, a + 8u, a + 16u, a + 24u, b, b + 2u, b + 4u, b + 6u,
                                     F16 ? ptx::idesc_f16(128, BNT) : ptx::idesc_bf16(128, BNT),
                                     q > 0 ? 1u : (first ^ 1u));
            }
          }
          first = 0;
          ptx::mma_commit_elect(&aempty[cur.slot]);   // frees the stage's A columns
        }
        if (!alive) break;
        ptx::mma_commit_elect(&xempty[rx.slot]);      // every issuer releases every X slot
        rx.next(SX);
      }
      g0 += uint32_t(nst);
      if (!alive) break;
      ptx::mma_commit_elect(&accfull[acc]);      // every issuer arrives once per unit
    }
    // Every MMA issued above has completed once `drain` flips.
    ptx::mma_commit_elect(drain);
    volatile int no_abort = 0;
    warp_all(ptx::mbar_wait(drain, 0, &no_abort, 200000000ull));
  } else if (A4 && warp < kEpiWarp0) {
    // ---------------------------------------------------------------- scale factors (A4)
    // One warpgroup, every stage: thread r (lane l = r % 32 of lane quarter r / 32) copies
    // into the stage's scale-factor columns
    //  - weight row r's four E8M0 bytes (the record's tail): the MMA reads row r's factors
    //    from lane r, column r / 32 of the group (the word is written to all four);
    //  - the activation scale words of tokens l, l + 32, l + 64, ...: the MMA reads token
    //    n's factors from lane n % 32, column n / 32, in every lane quarter (each quarter
    //    holds the same copy), as a probe with one marked exponent per call showed.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t t_lane = tbase + (uint32_t((warp & 3) * 32) << 16);
    constexpr int kTokGroups = (BNT + 127) / 128;            // groups of 4 token columns
    uint32_t g = 0;
    bool alive = true;
    Ring rx;                                             // the X ring, as the issuers walk it
    Unit w;
    int e_hint = -1;
    for (int uj = 0; alive && unit_at(uj, a, sc, BNT, prefix, offs, e_hint, w); ++uj) {
      const int nst = w.kb1 - w.kb0;
      for (int x0 = 0; x0 < nst && alive; x0 += XQ) {
        // the activation exponents of these stages arrive with the slot's codes
        if (!warp_all(ptx::mbar_wait(&xfull[rx.slot], rx.phase, abort_flag, T, kSleepDequant))) { alive = false; break; }
        const uint8_t* ex = s_x + rx.slot * C::kXSlotBytes + XQ * C::kXBytes;
        const int x1 = x0 + XQ < nst ? x0 + XQ : nst;
        for (int i = x0; i < x1; ++i, ++g) {
          const int kb = w.kb0 + i;
          uint32_t sfb[4 * kTokGroups];
#pragma unroll
          for (int c = 0; c < 4 * kTokGroups; ++c) {
            const int j = c * 32 + lane;                 // token of column c in this lane
            sfb[c] = j < BNT ? *reinterpret_cast<const uint32_t*>(
                                   ex + (i - x0) * C::kXExpBytes + j * 16 + (kb & 3) * 4)
                             : 0x7F7F7F7Fu;              // past the tile (zero codes anyway)
          }
          const int rs = int(g % uint32_t(SR)), ca = int(g % uint32_t(SA));
          if (!warp_all(ptx::mbar_wait(&rfull[rs], (g / uint32_t(SR)) & 1u, abort_flag, T, kSleepDequant))) { alive = false; break; }
          const uint32_t sfa = *reinterpret_cast<const uint32_t*>(s_rec + rs * C::kRecSlot + kCodeBytes + r * 4);
          ptx::fence_proxy_async_smem();                 // the reads above before the refills
          if (!warp_all(ptx::mbar_wait(&aempty[ca], ((g / uint32_t(SA)) & 1u) ^ 1u, abort_flag, T, kSleepDequant))) { alive = false; break; }
          ptx::tc_fence_after();
          const uint32_t col = t_lane + uint32_t(C::kACol0 + ca * C::kACols);
          ptx::tmem_st4(col, sfa, sfa, sfa, sfa);
#pragma unroll
          for (int h = 0; h < kTokGroups; ++h)
            ptx::tmem_st4(col + 4u + 4u * h, sfb[4 * h], sfb[4 * h + 1], sfb[4 * h + 2], sfb[4 * h + 3]);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          warp_arrive(&afull[ca], lane);
        }
        rx.next(SX);
      }
    }
  } else if (N8 && warp < kEpiWarp0) {
    // ---------------------------------------------------------------- scale factors (N8)
    // One warpgroup, every stage: thread r copies weight row r's four E8M0 bytes (the
    // stage's scale tail) into the stage's four scale-factor columns of lane r, as for the
    // register-decoded FP8 path; the activation side is the constant set in the prologue.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t t_lane = tbase + (uint32_t((warp & 3) * 32) << 16);
    uint32_t g = 0;
    bool alive = true;
    Unit w;
    int e_hint = -1;
    for (int uj = 0; alive && unit_at(uj, a, sc, BNT, prefix, offs, e_hint, w); ++uj) {
      const int nst = w.kb1 - w.kb0;
      for (int i = 0; i < nst; ++i, ++g) {
        const int rs = int(g % uint32_t(SR)), ca = int(g % uint32_t(SA));
        if (!warp_all(ptx::mbar_wait(&rfull[rs], (g / uint32_t(SR)) & 1u, abort_flag, T, kSleepDequant))) { alive = false; break; }
        const uint32_t sfa = *reinterpret_cast<const uint32_t*>(s_tail + rs * C::kTailBytes + r * 4);
        ptx::fence_proxy_async_smem();                 // the read above before the refill
        if (!warp_all(ptx::mbar_wait(&aempty[ca], ((g / uint32_t(SA)) & 1u) ^ 1u, abort_flag, T, kSleepDequant))) { alive = false; break; }
        ptx::tc_fence_after();
        ptx::tmem_st4(t_lane + uint32_t(C::kSfaCol0 + 4 * ca), sfa, sfa, sfa, sfa);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        warp_arrive(&afull[ca], lane);
      }
    }
  } else if (!kDirect && warp < kEpiWarp0) {
    // ---------------------------------------------------------------- dequant (2 WGs)
    const int wg = warp >> 2;                              // takes the stages g % kDeqWGs == wg
    const int r = (warp & 3) * 32 + lane;                  // weight row = TMEM lane
    const uint32_t t_lane = tbase + (uint32_t((warp & 3) * 32) << 16);
    const int G = L.groups_per_record;
    const int zoff = L.off_zeros - L.off_scales;
    uint32_t g0 = 0;                                       // CTA stage counter at the unit start
    bool alive = true;
    Unit w;
    int e_hint = -1;
    for (int uj = 0; alive && unit_at(uj, a, sc, BNT, prefix, offs, e_hint, w); ++uj) {
      const int nst = (w.kb1 - w.kb0) * kSub;
      // FP16 operands: the unit's expert's scale factor 2^k, from its packed header
      float w_pre = 1.0f;
      if constexpr (F16)
        w_pre = __ldg(&reinterpret_cast<const PackedHeader*>(
                          a.packed + int64_t(w.expert) * a.expert_stride)->w_prescale);
      // Visit only this warpgroup's stages; ring slots and phases follow from the stage
      // counter (the ring depths are compile-time constants).
      const uint32_t g1 = g0 + uint32_t(nst);
      uint32_t g = g0 + (uint32_t(wg) + uint32_t(kDeqWGs) - g0 % uint32_t(kDeqWGs)) % uint32_t(kDeqWGs);
      g0 = g1;
      for (; g < g1; g += uint32_t(kDeqWGs)) {
        const int i = int(g - (g1 - uint32_t(nst)));       // stage index inside the unit
        Ring cr, ca;
        cr.slot = int(g % uint32_t(SR));
        cr.phase = (g / uint32_t(SR)) & 1u;
        ca.slot = int(g % uint32_t(SA));
        ca.phase = (g / uint32_t(SA)) & 1u;
        if (!warp_all(ptx::mbar_wait(&rfull[cr.slot], cr.phase, abort_flag, T, kSleepDequant))) { alive = false; break; }
        const uint8_t* rec = s_rec + cr.slot * C::kRecSlot;
        const uint32_t a_col = t_lane + uint32_t(C::kACol0 + ca.slot * C::kACols);
        if constexpr (A8) {
          uint32_t regs[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 q = *reinterpret_cast<const uint4*>(rec + c * (kTileN * 16) + r * 16);
            const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
              decode_e2m1_to_e4m3_word(wd[j], regs[8 * c + 2 * j], regs[8 * c + 2 * j + 1]);
          }
          const uint32_t sf = *reinterpret_cast<const uint32_t*>(rec + kTail + r * 4);
          release_to_async(&rempty[cr.slot], lane);           // record consumed
          if (!warp_all(ptx::mbar_wait(&aempty[ca.slot], ca.phase ^ 1u, abort_flag, T, kSleepDequant))) { alive = false; break; }
          ptx::tc_fence_after();
          ptx::tmem_st4(t_lane + uint32_t(C::kSfaCol0 + 4 * ca.slot), sf, sf, sf, sf);
          ptx::tmem_st32(a_col, regs);
        } else {
          // A half record holds record chunks 2h, 2h + 1 (h = i % 2) in slot chunks 0, 1.
          const int rbase = (CH == 4) ? 0 : 2 * (i & 1);
          uint32_t regs[32];
          decode_two_chunks_a16<DM>(rec, kTail, 0, rbase, r, L.has_zp, G, zoff, w_pre, regs);
          if (CH == 2) release_to_async(&rempty[cr.slot], lane);
          if (!warp_all(ptx::mbar_wait(&aempty[ca.slot], ca.phase ^ 1u, abort_flag, T, kSleepDequant))) { alive = false; break; }
          ptx::tc_fence_after();
          ptx::tmem_st32(a_col, regs);
          if (CH == 4) {
            decode_two_chunks_a16<DM>(rec, kTail, 2, 2, r, L.has_zp, G, zoff, w_pre, regs);
            release_to_async(&rempty[cr.slot], lane);
            ptx::tmem_st32(a_col + 32u, regs);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        warp_arrive(&afull[ca.slot], lane);
      }
    }
  } else if (warp < kEpiWarp0 + RO::kEpiWarps) {
    // ---------------------------------------------------------------- epilogue
    // Warp e covers tensor-memory lanes 32 (e % 4) ... (its 32 weight rows) and the
    // accumulator columns (tokens) [eh * kCols, (eh + 1) * kCols) of its column half eh.
    constexpr int kHalves = RO::kEpiWarps / 4;
    constexpr int kCols = BNT / kHalves;
    constexpr int kChunk = kCols < 32 ? kCols : 32;
    const int eh = (warp - kEpiWarp0) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t t_lane = tbase + (uint32_t((warp & 3) * 32) << 16);
    uint32_t epi_phase = 0;
    // Bounded rendezvous of the epilogue threads (a named barrier could not give up).
    auto epi_sync = [&]() -> bool {
      warp_arrive(epibar, lane);
      const bool ok = ptx::mbar_wait(epibar, epi_phase, abort_flag, T, kSleepEpilogue);
      epi_phase ^= 1u;
      return warp_all(ok);
    };
    // This warp's accumulator chunk c (kChunk columns), partial accumulators summed in the
    // order sub0, sub0 + 1, ... (16 columns at a time, so that few registers are live).
    auto load_chunk = [&](int acc, int sub0, int active, int c, uint32_t (&v)[32]) {
      const uint32_t col = t_lane + uint32_t(acc * C::kNumSub * BNT + eh * kCols + c * kChunk);
#pragma unroll
      for (int h = 0; h < kChunk / 16; ++h) {
        uint32_t p16[16];
        ptx::tmem_ld16(col + uint32_t(sub0 * BNT + h * 16), p16);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[h * 16 + j] = p16[j];
#pragma unroll
        for (int d = 1; d < C::kNumSub; ++d) {
          if (d >= active) break;
          const int sub = (sub0 + d) % C::kNumSub;
          ptx::tmem_ld16(col + uint32_t(sub * BNT + h * 16), p16);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            v[h * 16 + j] = __float_as_uint(__uint_as_float(v[h * 16 + j]) + __uint_as_float(p16[j]));
        }
      }
    };
    int ui = 0;
    uint32_t g = 0;                       // stage counter of this CTA at the unit's start
    Unit w;
    int e_hint = -1;
    // Bias of output column n for the unit's expert (added after every scale).
    auto bias_of = [&](const Unit& u, int64_t n, bool n_ok) -> float {
      return (n_ok && a.bias != nullptr) ? __ldg(a.bias + int64_t(u.expert) * a.bias_stride + n)
                                         : 0.0f;
    };
    // Per-token activation scale of output row m (indexed: of the row it was gathered from).
    auto tok_scale_of = [&](int64_t m) -> float {
      if constexpr (GATHER) {
        const int t = __ldg(a.row_index + m);
        return t >= 0 && t < a.x_rows ? a.tok_scale[t] : 0.0f;
      }
      return a.tok_scale[m];
    };
    if constexpr (F16) ptx::grid_dependency_wait();   // the row scales come from the pre-pass
    for (int uj = 0; unit_at(uj, a, sc, BNT, prefix, offs, e_hint, w); ++uj, ++ui) {
      const int acc = ui % C::kNumAcc;
      const uint32_t acc_par = uint32_t((ui / C::kNumAcc) & 1);
      const int nst = (w.kb1 - w.kb0) * kSub;
      const uint32_t g0 = g;
      g += uint32_t(nst);
      if (!warp_all(ptx::mbar_wait(&accfull[acc], acc_par, abort_flag, T, kSleepEpilogue))) break;
      ptx::tc_fence_after();
      const int64_t n = int64_t(w.nt) * kTileN + r;
      const bool n_ok = n < L.N;
      const bool split = w.ncontrib > 1;
      __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.Y);
      // NVFP4 and the FP16 operands: the accumulator scale of the unit's expert, from its
      // packed header
      float acc_s = 1.0f;
      if constexpr (DM == DM_MXFP4_F16)     // (the header's acc_scale serves the BF16 decode)
        acc_s = 1.0f / __ldg(&reinterpret_cast<const PackedHeader*>(
                                a.packed + int64_t(w.expert) * a.expert_stride)->w_prescale);
      else if constexpr (DM == DM_NVFP4_F16)  // g 2^8 of the BF16 decode -> g 2^-4 (weights x 16)
        acc_s = 0x1p-12f * __ldg(&reinterpret_cast<const PackedHeader*>(
                                     a.packed + int64_t(w.expert) * a.expert_stride)->acc_scale);
      else if constexpr (DM == DM_NVFP4 || F16)
        acc_s = __ldg(&reinterpret_cast<const PackedHeader*>(
                          a.packed + int64_t(w.expert) * a.expert_stride)->acc_scale);
      // Partial accumulators of the issuers that had a stage in this unit: the unit's
      // stages g0, g0 + 1, ... went to issuers (g0 + d) % kIssuers.
      const int active = min(C::kNumSub, nst);
      const int sub0 = int(g0 % uint32_t(C::kNumSub));
      if constexpr (kHalves > 1) {
        if (!split) {
          // Wide tiles: scale and round every column of this warp to BF16 in registers,
          // hand the accumulator back to the MMA at once, then store.
          float cs = (n_ok && a.chan_scale != nullptr) ? a.chan_scale[n] : 1.0f;
          if constexpr (DM == DM_NVFP4 || F16) cs *= acc_s;
          uint32_t packed[kCols / 2];
          const bool with_bias = a.bias != nullptr;
          if (!with_bias) {
            // the accumulator is read, scaled by c[n] and rounded; the per-token scale comes
            // after the release below (FP16 operands: a power of two, which commutes with the
            // rounding; FP8: a second rounding, within that path's tolerance)
#pragma unroll
            for (int c = 0; c < kCols / 16; ++c) {
              uint32_t v[16];
              ptx::tmem_ld16(t_lane + uint32_t(acc * C::kNumSub * BNT + eh * kCols + c * 16), v);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; j += 2)
                packed[(c * 16 + j) / 2] =
                    ptx::pack_bf16x2(__uint_as_float(v[j]) * cs, __uint_as_float(v[j + 1]) * cs);
            }
          } else {
            // with a bias every scale comes before the single rounding: the per-token scales
            // of this warp's columns are held one per lane (column l + 32 i in lane l; never
            // gathered rows here) and handed out by shuffles
            const float b = bias_of(w, n, n_ok);
            float tk[kCols / 32];
#pragma unroll
            for (int i = 0; i < kCols / 32; ++i) {
              const int64_t m = w.row0 + int64_t(eh) * kCols + i * 32 + lane;
              tk[i] = (kTokScale && m < w.row_end) ? a.tok_scale[m] : 1.0f;
            }
#pragma unroll
            for (int c = 0; c < kCols / 16; ++c) {
              uint32_t v[16];
              ptx::tmem_ld16(t_lane + uint32_t(acc * C::kNumSub * BNT + eh * kCols + c * 16), v);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                float y0 = __uint_as_float(v[j]) * cs, y1 = __uint_as_float(v[j + 1]) * cs;
                if constexpr (kTokScale) {
                  const int col = c * 16 + j;
                  y0 *= __shfl_sync(0xffffffffu, tk[col / 32], col % 32);
                  y1 *= __shfl_sync(0xffffffffu, tk[(col + 1) / 32], (col + 1) % 32);
                }
                packed[(c * 16 + j) / 2] = ptx::pack_bf16x2(y0 + b, y1 + b);
              }
            }
          }
          ptx::tc_fence_before();
          warp_arrive(&accempty[acc], lane);
          if (n_ok) {
            uint16_t* Yh = reinterpret_cast<uint16_t*>(Y) + n;
#pragma unroll
            for (int j = 0; j < kCols; ++j) {
              const int64_t m = w.row0 + int64_t(eh) * kCols + j;   // (never a gathered tile)
              if (m < w.row_end) {
                uint16_t h = uint16_t(j & 1 ? packed[j / 2] >> 16 : packed[j / 2] & 0xFFFFu);
                if (kTokScale && !with_bias)
                  h = uint16_t(ptx::pack_bf16x2(__uint_as_float(uint32_t(h) << 16) * a.tok_scale[m],
                                                0.0f) & 0xFFFFu);
                Yh[m * a.ldy] = h;
              }
            }
          }
          continue;
        }
      }
      if (!split) {
        // Narrow tiles (double-buffered accumulators): convert and store chunk by chunk.
        float cs = (n_ok && a.chan_scale != nullptr) ? a.chan_scale[n] : 1.0f;
        if constexpr (DM == DM_NVFP4 || F16) cs *= acc_s;
        const float b = bias_of(w, n, n_ok);
#pragma unroll 1
        for (int c = 0; c < kCols / kChunk; ++c) {
          uint32_t v[32];
          load_chunk(acc, sub0, active, c, v);
          if (c == kCols / kChunk - 1) {
            ptx::tc_fence_before();
            warp_arrive(&accempty[acc], lane);
          }
          if (n_ok) {
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
              const int64_t m = w.row0 + int64_t(eh) * kCols + c * kChunk + j;
              if (m < w.row_end) {
                float y = __uint_as_float(v[j]) * cs;
                if (kTokScale) y *= tok_scale_of(m);
                Y[m * a.ldy + n] = __float2bfloat16_rn(y + b);
              }
            }
          }
        }
        continue;
      }
      // Cut tile: store this contributor's FP32 partial tile into its slot of the
      // workspace (row r of the slot is kTileN-major: BNT contiguous floats per weight row).
      const int64_t slot_floats = int64_t(kTileN) * BNT;
      float* my_row = a.ws + int64_t(w.slot0 + w.contrib) * slot_floats + int64_t(r) * BNT +
                      eh * kCols;
#pragma unroll 1
      for (int c = 0; c < kCols / kChunk; ++c) {
        uint32_t v[32];
        load_chunk(acc, sub0, active, c, v);
        if (c == kCols / kChunk - 1) {
          ptx::tc_fence_before();
          warp_arrive(&accempty[acc], lane);
        }
#pragma unroll
        for (int j = 0; j < kChunk; j += 4)
          __stcg(reinterpret_cast<float4*>(my_row + c * kChunk + j),
                 make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                             __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])));
      }
      // The last contributor to arrive sums the slots and converts.
      __threadfence();
      if (!epi_sync()) break;
      if (r == 0 && eh == 0) {
        const int prev = atomicAdd(&a.counters[w.tile_id], 1);
        misc[4] = (prev == w.ncontrib - 1) ? 1 : 0;
        if (prev == w.ncontrib - 1) a.counters[w.tile_id] = 0;
      }
      if (!epi_sync()) break;
      if (misc[4]) {
        // Sum in contributor order (fixed by the schedule, not by the arrival order), two
        // contributors' loads in flight at a time, 16 columns per pass.
        __threadfence();
        const float* row0p = a.ws + int64_t(w.slot0) * slot_floats + int64_t(r) * BNT +
                             eh * kCols;
        float cs2 = (n_ok && a.chan_scale != nullptr) ? a.chan_scale[n] : 1.0f;
        if constexpr (DM == DM_NVFP4 || F16) cs2 *= acc_s;
        const float b2 = bias_of(w, n, n_ok);
        constexpr int kPass = kCols < 16 ? kCols : 16;
#pragma unroll 1
        for (int c0 = 0; c0 < kCols; c0 += kPass) {
          float sum[kPass];
#pragma unroll
          for (int j = 0; j < kPass; ++j) sum[j] = 0.0f;
#pragma unroll 2
          for (int q = 0; q < w.ncontrib; ++q) {
            const float4* src = reinterpret_cast<const float4*>(row0p + q * slot_floats + c0);
#pragma unroll
            for (int j = 0; j < kPass / 4; ++j) {
              const float4 x = __ldcg(src + j);
              sum[4 * j] += x.x;
              sum[4 * j + 1] += x.y;
              sum[4 * j + 2] += x.z;
              sum[4 * j + 3] += x.w;
            }
          }
          if (n_ok) {
#pragma unroll
            for (int j = 0; j < kPass; ++j) {
              const int64_t m = w.row0 + int64_t(eh) * kCols + c0 + j;
              if (m < w.row_end) {
                float y = sum[j] * cs2;
                if (kTokScale) y *= tok_scale_of(m);
                Y[m * a.ldy + n] = __float2bfloat16_rn(y + b2);
              }
            }
          }
        }
      }
      if (!epi_sync()) break;
    }
  }

  // ------------------------------------------------------------------ teardown
  // (the abort flag is read after the barrier: a role that finished early must not miss
  // a wait that gave up later in another role)
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) atomicCAS(a.status, 0, kStatusTimeout);
  if (warp == kEpiWarp0) ptx::tmem_dealloc(tbase, C::kTmemCols);
}

template <int BNT, bool A8, int DM, bool GATHER>
cudaError_t launch_variant(const GemmPlan& plan, const CUtensorMap& tmap, const GemmArgs& args,
                           cudaStream_t st) {
  using C = GemmCfg<BNT, A8, DM == DM_W4A4, DM == DM_W4A8N>;
  // At least 120 KB of shared memory per CTA: one CTA per SM, so no CTA ever waits for
  // another one's tensor-memory allocation.
  constexpr int kSmem = C::kSmemBytes > 120 * 1024 ? C::kSmemBytes : 120 * 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(qgemm_tc_kernel<BNT, A8, DM, GATHER>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(plan.grid));
  cfg.blockDim = dim3(Roles<BNT, DM == DM_W4A4 || DM == DM_W4A8N, A8>::kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = plan.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, qgemm_tc_kernel<BNT, A8, DM, GATHER>, tmap, args);
}

template <bool A8, int DM>
cudaError_t launch_gemm_impl(const GemmPlan& plan, const CUtensorMap& tmap, const GemmArgs& args,
                             cudaStream_t st) {
  if (args.row_index != nullptr) {          // gathered (indexed MoE) tiles: up to 64 tokens
    if constexpr (DM == DM_W4A4) return cudaErrorInvalidValue;   // W4A4: TMA loads only
    else switch (plan.token_tile) {
      case 16: return launch_variant<16, A8, DM, true>(plan, tmap, args, st);
      case 32: return launch_variant<32, A8, DM, true>(plan, tmap, args, st);
      case 64: return launch_variant<64, A8, DM, true>(plan, tmap, args, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (plan.token_tile) {
    case 16: return launch_variant<16, A8, DM, false>(plan, tmap, args, st);
    case 32: return launch_variant<32, A8, DM, false>(plan, tmap, args, st);
    case 64: return launch_variant<64, A8, DM, false>(plan, tmap, args, st);
    case 128: return launch_variant<128, A8, DM, false>(plan, tmap, args, st);
    case 256: return launch_variant<256, A8, DM, false>(plan, tmap, args, st);
    default: return cudaErrorInvalidValue;
  }
}

// Decode mode of a packed layout (BF16 activations).
inline int decode_mode(const Layout& L) {
  if (L.afmt == A_MXFP4) return DM_W4A4;
  if (L.afmt == A_FP8N) return DM_W4A8N;
  if (L.wfmt == W_MXFP4) return DM_MXFP4;
  if (L.wfmt == W_MXINT4) return DM_MXINT4;
  if (L.wfmt == W_NVFP4) return DM_NVFP4;
  if (L.groups_per_record == 1) return L.has_zp ? DM_INT4_ZP_G1 : DM_INT4_SYM_G1;
  return DM_INT4_ANY;
}

template <bool A8>
int x_box_slabs_impl(int bnt) {
  switch (bnt) {
    case 16: return GemmCfg<16, A8>::kXBoxSlabs;
    case 32: return GemmCfg<32, A8>::kXBoxSlabs;
    case 64: return GemmCfg<64, A8>::kXBoxSlabs;
    case 128: return GemmCfg<128, A8>::kXBoxSlabs;
    case 256: return GemmCfg<256, A8>::kXBoxSlabs;
    default: return -1;
  }
}

template <bool A8>
int smem_bytes_impl(int bnt) {
  switch (bnt) {
    case 16: return GemmCfg<16, A8>::kSmemBytes;
    case 32: return GemmCfg<32, A8>::kSmemBytes;
    case 64: return GemmCfg<64, A8>::kSmemBytes;
    case 128: return GemmCfg<128, A8>::kSmemBytes;
    case 256: return GemmCfg<256, A8>::kSmemBytes;
    default: return -1;
  }
}

}  // namespace qgemm
