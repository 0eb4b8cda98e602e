// The tcgen05 quantized-weight GEMM kernel (dense and MoE grouped), sm_103a.
//
// Design (one persistent CTA per SM, warp-specialised):
//   warp 0     producer: per pipeline stage, one TMA 2-D tile of X (token_tile rows x
//              128 bytes, 128-byte swizzle) plus bulk copies of the packed weight tile
//              (128 rows x BK K-elements, 4 bits each), its scale tile and zero-point tile;
//              all complete on the stage's `full` mbarrier.
//   warps 2-5  dequant: thread r owns weight row r (= tensor-memory lane r).  It decodes
//              its row's BK codes in registers (dequant.cuh) and stores them with
//              tcgen05.st into the stage's A-operand columns of tensor memory.  The
//              dequantized weights never touch shared memory, which stays free for the
//              activation operand.
//   warp 1     MMA issuer (one thread): tcgen05.mma with A = weights in tensor memory
//              (M = 128 weight rows), B = activation tile in shared memory (N = token_tile
//              rows of X), accumulating FP32 in tensor memory (the "swap-AB" orientation:
//              the weights fill the 128-row side, so small batches still run full-height
//              MMAs).  BF16 activations use kind::f16; FP8 activations use
//              kind::mxf8f6f4 with the E8M0 weight scales as block scale factors.
//   warps 6-9  epilogue: tcgen05.ld of the accumulator, fused per-channel / per-token
//              scaling, BF16 store of Y (or FP32 split-K reduction through a workspace;
//              the last CTA of a tile converts and re-zeroes the workspace).
// Data-dependent parts of the pages this follows: "Humming wird angekündigt", sections
// "Gemeinsam genutzte CUDA-Komponenten" (task scheduling, data movement with TMA,
// dequantization and scaling fused into the kernel, tensor-core compute, output stage
// with fused scaling; dense vs MoE scheduling), "Leistungsoptimierung basierend auf
// Geräteparametern" (fast MXFP4 -> FP8 conversion for W4A8; Stream-K style scheduling).
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

constexpr int kThreads = 320;
constexpr int kMaxExperts = 1024;
constexpr int kScaleSlot = 512;      // bytes reserved per stage for a scale tile
constexpr int kZeroSlot = 128;       // bytes reserved per stage for a zero-point tile

template <int BNT, bool A8>
struct GemmCfg {
  static constexpr int kStageK = A8 ? 128 : 64;                  // K-elements per stage
  static constexpr int kActBytes = BNT * 128;                      // one 128-byte row per token
  static constexpr int kCodeBytes = kTileN * kStageK / 2;
  static constexpr int kNumAcc = (BNT <= 128) ? 2 : 1;
  static constexpr int kStages = BNT >= 256 ? 5 : (BNT >= 128 ? (A8 ? 6 : 8) : (BNT >= 64 ? 10 : 12));
  static constexpr int kAccCols = kNumAcc * BNT;
  static constexpr int kACol0 = (kAccCols + 31) / 32 * 32;
  // Block-scale factors (FP8 activations only): per stage one 4-column slot for the
  // weight-side factors (a row's four E8M0 bytes, one per 32 K, replicated over the four
  // columns of its lane), then 8 columns holding the constant activation-side factor.
  static constexpr int kSfaCol0 = kACol0 + kStages * 32;
  static constexpr int kSfbCol0 = (kSfaCol0 + (A8 ? 4 * kStages : 0) + 7) / 8 * 8;
  static constexpr int kUsedCols = kSfbCol0 + (A8 ? 8 : 0);
  static constexpr int kTmemCols = kUsedCols <= 32 ? 32 : kUsedCols <= 64 ? 64 :
                                   kUsedCols <= 128 ? 128 : kUsedCols <= 256 ? 256 : 512;
  static_assert(kUsedCols <= 512, "tensor memory budget");
  static constexpr int kStageBytes = kActBytes + kCodeBytes + kScaleSlot + kZeroSlot;
  static constexpr int kBarBytes = (3 * kStages + 2 * kNumAcc + 2) * 8;
  static constexpr int kMiscBytes = 64 + 2 * (kMaxExperts + 1) * 4;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes + kMiscBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct Unit {
  int nt, mt, split, expert;
  int kb0, kb1;
  int64_t row0, row_end;
};

__device__ __forceinline__ Unit decode_unit(int u, const GemmArgs& a, int bnt, const int* prefix,
                                            const int* offs) {
  Unit w;
  const int n_tiles = int(a.L.n_tiles);
  const int k_blocks = int(a.L.k_blocks);
  if (a.offsets == nullptr) {
    w.split = u % a.splits;
    const int tile = u / a.splits;
    w.nt = tile % n_tiles;
    w.mt = tile / n_tiles;
    w.expert = 0;
    w.row0 = int64_t(w.mt) * bnt;
    w.row_end = a.M;
    w.kb0 = int(int64_t(w.split) * k_blocks / a.splits);
    w.kb1 = int(int64_t(w.split + 1) * k_blocks / a.splits);
  } else {
    w.nt = u % n_tiles;
    const int gmt = u / n_tiles;
    int lo = 0, hi = a.E;                    // largest e with prefix[e] <= gmt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= gmt) lo = mid; else hi = mid;
    }
    w.expert = lo;
    w.mt = gmt - prefix[lo];
    w.split = 0;
    w.row0 = int64_t(offs[lo]) + int64_t(w.mt) * bnt;
    w.row_end = offs[lo + 1];
    w.kb0 = 0;
    w.kb1 = k_blocks;
  }
  return w;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

template <int BNT, bool A8>
__global__ void __launch_bounds__(kThreads, 1)
qgemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const GemmArgs a) {
  using C = GemmCfg<BNT, A8>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_act = smem;
  uint8_t* s_code = s_act + S * C::kActBytes;
  uint8_t* s_scale = s_code + S * C::kCodeBytes;
  uint8_t* s_zero = s_scale + S * kScaleSlot;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_zero + S * kZeroSlot);
  uint64_t* afull = full + S;
  uint64_t* empty = afull + S;
  uint64_t* accfull = empty + S;
  uint64_t* accempty = accfull + C::kNumAcc;
  uint64_t* drain = accempty + C::kNumAcc;
  uint64_t* epibar = drain + 1;                    // epilogue-warps rendezvous (split-K)
  int* misc = reinterpret_cast<int*>(epibar + 1);  // [0] tmem base [1] abort [2] ok [3] units
  int* prefix = misc + 16;                         // MoE: m-tiles before expert e
  int* offs = prefix + (kMaxExperts + 1);          // MoE: row offsets

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Layout& L = a.L;

  // ------------------------------------------------------------------ prologue
  if (threadIdx.x == 0) {
    misc[1] = 0;
    const PackedHeader* h = reinterpret_cast<const PackedHeader*>(a.packed);
    bool ok = h->magic == kPackedMagic && h->version == kPackedVersion && h->wfmt == L.wfmt &&
              h->group == L.group && h->has_zp == L.has_zp && h->afmt == L.afmt &&
              h->N == L.N && h->K == L.K && h->total_bytes == L.total_bytes;
    if (ok && a.offsets != nullptr && a.E > 1) {
      const PackedHeader* hl =
          reinterpret_cast<const PackedHeader*>(a.packed + int64_t(a.E - 1) * a.expert_stride);
      ok = hl->magic == kPackedMagic && hl->N == L.N && hl->K == L.K && hl->afmt == L.afmt;
    }
    if (!ok) atomicCAS(a.status, 0, kStatusBadPacked);
    misc[2] = ok ? 1 : 0;
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&afull[s], 128);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < C::kNumAcc; ++i) {
      ptx::mbar_init(&accfull[i], 1);
      ptx::mbar_init(&accempty[i], 128);
    }
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(epibar, 128);
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) ptx::prefetch_tmap(&tmap_x);
  int num_units = a.num_units;
  if (a.offsets != nullptr && warp == 2) {
    // MoE schedule: m-tiles per expert and their exclusive prefix (one warp).
    int carry = 0;
    bool bad = false;
    for (int base = 0; base <= a.E; base += 32) {
      const int e = base + lane;
      int o = 0, t = 0;
      if (e <= a.E) {
        o = a.offsets[e];
        offs[e] = o;
      }
      if (e < a.E) {
        const int o1 = a.offsets[e + 1];
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
  __syncthreads();
  if (a.offsets != nullptr) num_units = misc[3] * int(L.n_tiles);
  if (!misc[2] || int(blockIdx.x) >= num_units) return;     // nothing allocated yet

  if (warp == 1) {
    ptx::tmem_alloc(reinterpret_cast<uint32_t*>(&misc[0]), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = static_cast<uint32_t>(misc[0]);
  volatile int* abort_flag = &misc[1];
  const uint64_t T = a.timeout_ns;

  if (A8 && warp >= 6) {
    // Activation-side block scale: a constant 2^6 (E8M0 133) that returns the factor 2^-6
    // of the e2m1 -> e4m3 byte shuffle.  Filled over every lane of its columns.
    const uint32_t tl = tbase + (uint32_t((warp & 3) * 32) << 16);
    ptx::tmem_st4(tl + C::kSfbCol0, 0x85858585u, 0x85858585u, 0x85858585u, 0x85858585u);
    ptx::tmem_st4(tl + C::kSfbCol0 + 4, 0x85858585u, 0x85858585u, 0x85858585u, 0x85858585u);
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_parity[S];
      bool issued[S];
      for (int s = 0; s < S; ++s) issued[s] = false;
      bool alive = true;
      for (int u = blockIdx.x; u < num_units && alive; u += gridDim.x) {
        const Unit w = decode_unit(u, a, BNT, prefix, offs);
        const uint8_t* P = a.packed + int64_t(w.expert) * a.expert_stride;
        const uint8_t* codes = P + L.off_codes + int64_t(w.nt) * L.k_blocks * L.code_tile_bytes;
        const int64_t st_base = int64_t(w.nt) * L.scale_tiles;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, T)) { alive = false; break; }
          const int64_t stile = L.groups_per_tile == 1 ? (int64_t(kb) * C::kStageK) / L.group : kb;
          const uint32_t bytes = uint32_t(C::kActBytes + L.code_tile_bytes + L.scale_tile_bytes +
                                          (L.has_zp ? L.zero_tile_bytes : 0));
          ptx::mbar_arrive_expect_tx(&full[stage], bytes);
          ptx::tma_load_2d(s_act + stage * C::kActBytes, &tmap_x, kb * C::kStageK,
                           int32_t(w.row0), &full[stage]);
          ptx::bulk_g2s(s_code + stage * C::kCodeBytes, codes + int64_t(kb) * L.code_tile_bytes,
                        uint32_t(L.code_tile_bytes), &full[stage], pol_w);
          ptx::bulk_g2s(s_scale + stage * kScaleSlot,
                        P + L.off_scales + (st_base + stile) * L.scale_tile_bytes,
                        uint32_t(L.scale_tile_bytes), &full[stage], pol_w);
          if (L.has_zp)
            ptx::bulk_g2s(s_zero + stage * kZeroSlot,
                          P + L.off_zeros + (st_base + stile) * L.zero_tile_bytes,
                          uint32_t(L.zero_tile_bytes), &full[stage], pol_w);
          issued[stage] = true;
          issued_parity[stage] = phase;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!alive) {
        // Wind down: let every copy this thread issued land before the CTA exits.
        volatile int no_abort = 0;
        for (int s = 0; s < S; ++s)
          if (issued[s]) ptx::mbar_wait(&full[s], issued_parity[s], &no_abort, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int ui = 0;
      bool alive = true;
      for (int u = blockIdx.x; u < num_units && alive; u += gridDim.x, ++ui) {
        const Unit w = decode_unit(u, a, BNT, prefix, offs);
        const int acc = ui % C::kNumAcc;
        const uint32_t acc_par = uint32_t((ui / C::kNumAcc) & 1);
        if (!ptx::mbar_wait(&accempty[acc], acc_par ^ 1u, abort_flag, T)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tbase + uint32_t(acc * BNT);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!ptx::mbar_wait(&afull[stage], phase, abort_flag, T)) { alive = false; break; }
          ptx::tc_fence_after();
          const uint64_t bdesc = ptx::desc_kmajor_sw128(ptx::smem_u32(s_act + stage * C::kActBytes));
          const uint32_t a_tmem = tbase + uint32_t(C::kACol0 + stage * 32);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t accum = (kb > w.kb0 || kk > 0) ? 1u : 0u;
            if constexpr (A8) {
              ptx::mma_mxf8f6f4_ts(d_tmem, a_tmem + kk * 8, bdesc + uint64_t(kk * 2),
                                   ptx::idesc_mxf8_e4m3(128, BNT, kk, 0),
                                   tbase + uint32_t(C::kSfaCol0 + 4 * stage),
                                   tbase + uint32_t(C::kSfbCol0), accum);
            } else {
              ptx::mma_f16_ts(d_tmem, a_tmem + kk * 8, bdesc + uint64_t(kk * 2),
                              ptx::idesc_bf16(128, BNT), accum);
            }
          }
          ptx::mma_commit(&empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!alive) break;
        ptx::mma_commit(&accfull[acc]);
      }
      // Every MMA issued above has completed once `drain` flips.
      ptx::mma_commit(drain);
      volatile int no_abort = 0;
      ptx::mbar_wait(drain, 0, &no_abort, 200000000ull);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- dequant
    const int r = (warp & 3) * 32 + lane;                  // weight row = TMEM lane
    const uint32_t t_lane = tbase + (uint32_t((warp & 3) * 32) << 16);
    int stage = 0;
    uint32_t phase = 0;
    const int G = L.groups_per_tile;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const Unit w = decode_unit(u, a, BNT, prefix, offs);
      bool alive = true;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        if (!warp_all(ptx::mbar_wait(&full[stage], phase, abort_flag, T))) { alive = false; break; }
        const uint8_t* cs = s_code + stage * C::kCodeBytes;
        const uint8_t* ss = s_scale + stage * kScaleSlot;
        uint32_t regs[32];
        if constexpr (A8) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 q = *reinterpret_cast<const uint4*>(cs + c * 2048 + r * 16);
            const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
              decode_e2m1_to_e4m3_word(wd[j], regs[8 * c + 2 * j], regs[8 * c + 2 * j + 1]);
          }
          const uint32_t sf = *reinterpret_cast<const uint32_t*>(ss + r * 4);   // 4 x E8M0
          ptx::tmem_st4(t_lane + uint32_t(C::kSfaCol0 + 4 * stage), sf, sf, sf, sf);
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint4 q = *reinterpret_cast<const uint4*>(cs + c * 2048 + r * 16);
            const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
            const int ge = (G == 1) ? 0 : c;                  // group entry of this chunk
            if (L.wfmt == W_MXFP4) {
              const uint32_t E = ss[r * G + ge];
              uint32_t sa, sb;
              bool big;
              mxfp4_factors(E, sa, sb, big);
              const bool two = __any_sync(0xffffffffu, big);
#pragma unroll
              for (int j = 0; j < 4; ++j) decode_mxfp4_word(wd[j], sa, sb, two, &regs[16 * c + 4 * j]);
            } else {
              const uint32_t s = reinterpret_cast<const uint16_t*>(ss)[r * G + ge];
              uint32_t z = 8;
              if (L.has_zp) {
                const int zi = r * G + ge;
                z = (s_zero[stage * kZeroSlot + (zi >> 1)] >> (4 * (zi & 1))) & 0xFu;
              }
              const uint32_t zz = (0x4300u | z) * 0x00010001u;
              const uint32_t s2 = s * 0x00010001u;
#pragma unroll
              for (int j = 0; j < 4; ++j) decode_int4_word(wd[j], zz, s2, &regs[16 * c + 4 * j]);
            }
          }
        }
        ptx::tmem_st32(t_lane + uint32_t(C::kACol0 + stage * 32), regs);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&afull[stage]);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!alive) break;
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int r = (warp & 3) * 32 + lane;
    const uint32_t t_lane = tbase + (uint32_t((warp & 3) * 32) << 16);
    uint32_t epi_phase = 0;
    // Bounded rendezvous of the 128 epilogue threads (a named barrier could not give up).
    auto epi_sync = [&]() -> bool {
      ptx::mbar_arrive(epibar);
      const bool ok = ptx::mbar_wait(epibar, epi_phase, abort_flag, T);
      epi_phase ^= 1u;
      return warp_all(ok);
    };
    int ui = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++ui) {
      const Unit w = decode_unit(u, a, BNT, prefix, offs);
      const int acc = ui % C::kNumAcc;
      const uint32_t acc_par = uint32_t((ui / C::kNumAcc) & 1);
      if (!warp_all(ptx::mbar_wait(&accfull[acc], acc_par, abort_flag, T))) break;
      ptx::tc_fence_after();
      const int64_t n = int64_t(w.nt) * kTileN + r;
      const bool n_ok = n < L.N;
      const bool split = a.splits > 1;
      const float cs = (n_ok && a.chan_scale != nullptr && !split) ? a.chan_scale[n] : 1.0f;
      __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(a.Y);
      constexpr int kChunk = BNT < 32 ? BNT : 32;
#pragma unroll 1
      for (int c = 0; c < BNT / kChunk; ++c) {
        uint32_t v[32];
        if constexpr (kChunk == 32) {
          ptx::tmem_ld32(t_lane + uint32_t(acc * BNT + c * 32), v);
        } else {
          uint32_t v16[16];
          ptx::tmem_ld16(t_lane + uint32_t(acc * BNT), v16);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = v16[j];
        }
        ptx::tmem_wait_ld();
        if (c == BNT / kChunk - 1) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(&accempty[acc]);
        }
        if (n_ok) {
#pragma unroll
          for (int j = 0; j < kChunk; ++j) {
            const int64_t m = w.row0 + c * kChunk + j;
            if (m < w.row_end) {
              float y = __uint_as_float(v[j]);
              if (split) {
                ptx::red_add_f32(a.ws + m * a.ws_ld + n, y);
              } else {
                y *= cs;
                if (A8) y *= a.tok_scale[m];
                Y[m * a.ldy + n] = __float2bfloat16_rn(y);
              }
            }
          }
        }
      }
      if (split) {
        // Split-K: the last of the `splits` CTAs that reduce this tile converts it.
        __threadfence();
        if (!epi_sync()) break;
        if (r == 0) {
          const int tile = w.mt * int(L.n_tiles) + w.nt;
          const int prev = atomicAdd(&a.counters[tile], 1);
          misc[4] = (prev == a.splits - 1) ? 1 : 0;
          if (prev == a.splits - 1) a.counters[tile] = 0;
        }
        if (!epi_sync()) break;
        if (misc[4]) {
          __threadfence();
          if (n_ok) {
            const float cs2 = a.chan_scale != nullptr ? a.chan_scale[n] : 1.0f;
            const int64_t m_end = w.row0 + BNT < w.row_end ? w.row0 + BNT : w.row_end;
            for (int64_t m = w.row0; m < m_end; ++m) {
              float* p = a.ws + m * a.ws_ld + n;
              float y = __ldcg(p) * cs2;
              if (A8) y *= a.tok_scale[m];
              Y[m * a.ldy + n] = __float2bfloat16_rn(y);
              __stcg(p, 0.0f);
            }
          }
        }
        if (!epi_sync()) break;
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  if (threadIdx.x == 0 && *abort_flag) atomicCAS(a.status, 0, kStatusTimeout);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tbase, C::kTmemCols);
}

template <int BNT, bool A8>
cudaError_t launch_variant(const GemmPlan& plan, const CUtensorMap& tmap, const GemmArgs& args,
                           cudaStream_t st) {
  using C = GemmCfg<BNT, A8>;
  // At least 120 KB of shared memory per CTA: one CTA per SM, so no CTA ever waits for
  // another one's tensor-memory allocation.
  constexpr int kSmem = C::kSmemBytes > 120 * 1024 ? C::kSmemBytes : 120 * 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(qgemm_tc_kernel<BNT, A8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  qgemm_tc_kernel<BNT, A8><<<plan.grid, kThreads, kSmem, st>>>(tmap, args);
  return cudaGetLastError();
}

template <bool A8>
cudaError_t launch_gemm_impl(const GemmPlan& plan, const CUtensorMap& tmap, const GemmArgs& args,
                             cudaStream_t st) {
  switch (plan.token_tile) {
    case 16: return launch_variant<16, A8>(plan, tmap, args, st);
    case 32: return launch_variant<32, A8>(plan, tmap, args, st);
    case 64: return launch_variant<64, A8>(plan, tmap, args, st);
    case 128: return launch_variant<128, A8>(plan, tmap, args, st);
    case 256: return launch_variant<256, A8>(plan, tmap, args, st);
    default: return cudaErrorInvalidValue;
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
