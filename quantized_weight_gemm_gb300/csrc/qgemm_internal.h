// Internal definitions shared by the host dispatcher and the sm_103a kernels.
//
// Packed weight layout (one weight matrix; an MoE layer stacks E of them).  The repack
// pads N to a multiple of 128 (one tile of weight rows = the M side of the tensor-core
// instruction) and K to a multiple of 128 (one pipeline stage), then stores
//
//   [header: 256 B]
//   [record (n_tile 0, k_block 0)] [record (0, 1)] ... [record (n_tiles-1, k_blocks-1)]
//
// One record holds everything one pipeline stage needs, so the kernel fetches it with a
// single bulk copy:
//   codes  : [4 chunks][128 rows][16 B]; chunk c of row r holds K-elements 32c .. 32c+31
//            of that row as four 32-bit words of 8 nibbles, the nibbles interleaved so one
//            mask yields two decoded lanes (dequant.cuh); MXFP4 and NVFP4 weights for BF16
//            activations keep the natural order instead (element 2j in the low nibble of
//            byte j, the input of the hardware e2m1x2 conversion);
//            MXFP4 activations (W4A4): the tensor core reads the codes straight from shared
//            memory instead, so they are its operand layout -- K-major rows of 64 bytes
//            (128 K, element 2j in the low nibble of byte j), 8-row atoms of 512 bytes, the
//            16-byte piece c of row r at position c ^ ((r >> 1) & 3) of its row (the
//            64-byte swizzle);
//            FP8 activations on FP4 operands (A_FP8N): plain K-major rows of 64 bytes, the
//            same nibble order, row r at byte 64 r -- a tensor the TMA loads with its
//            "16 x 4-bit in 16 bytes" expansion, which writes the padded shared-memory
//            layout the block-scaled FP8/FP6/FP4 MMA reads e2m1 operands from;
//   scales : [128 rows][G] entries of S bytes, G = max(1, 128 / group) groups per record,
//            S = 2 (BF16) or 1 (E8M0, E4M3); a group longer than 128 repeats in each record;
//   zeros  : (INT4 with zero points only) [128 rows x G] nibbles, entry (r, j) in nibble
//            (r*G + j) & 1 of byte (r*G + j) / 2.
// Records are multiples of 16 bytes and the first starts 256 bytes in, so every record is
// one aligned bulk copy.
#pragma once

#include <stdint.h>

#ifndef __CUDACC__
#define __host__
#define __device__
#endif

namespace qgemm {

constexpr uint32_t kPackedMagic = 0x32575147u;   // "GQW2"
constexpr uint32_t kPackedVersion = 5;
constexpr int kTileN = 128;                      // weight rows per tile (MMA M)
constexpr int kStageK = 128;                     // K-elements per pipeline stage
constexpr int kCodeBytes = kTileN * kStageK / 2; // 8192
constexpr int kHeaderBytes = 256;

enum WFmt : int32_t { W_INT4_SYM = 0, W_UINT4_ZP = 1, W_MXFP4 = 2, W_MXINT4 = 3, W_NVFP4 = 4 };
// A_FP8N: FP8 activations with the e2m1 weights fed to the tensor core as FP4 operands
// (no register decode; see the codes layout above).
enum AFmt : int32_t { A_BF16 = 0, A_FP8 = 1, A_MXFP4 = 2, A_FP8N = 3 };

// Byte offset of the 16-byte piece (row r, 32-K chunk c) inside a record's codes.
inline __host__ __device__ int code_piece_offset(int32_t afmt, int r, int c) {
  return afmt == A_MXFP4 ? (r >> 3) * 512 + (r & 7) * 64 + ((c ^ ((r >> 1) & 3)) << 4)
         : afmt == A_FP8N ? r * 64 + c * 16
                          : c * (kTileN * 16) + r * 16;
}

struct PackedHeader {
  uint32_t magic;
  uint32_t version;
  int32_t wfmt, sdtype, group, has_zp, afmt, groups_per_record;
  int64_t N, K;
  int64_t n_tiles, k_blocks, record_bytes;
  int64_t off_scales, off_zeros, total_bytes;    // offsets inside a record / total size
  // Factor the GEMM applies to its FP32 accumulators (NVFP4: the per-tensor scale times
  // 2^8, the decode having left the weights 2^8 smaller; INT4 with BF16 scales: 2^-k, see
  // w_prescale; 1 for the other formats).
  float acc_scale;
  // INT4 with BF16 scales: the power of two 2^k that the decode multiplies every scale by
  // before rounding the weight to FP16, chosen from the largest |scale| of the tensor so
  // that (q - z) * s * 2^k stays inside FP16's normal range.  MXFP4 (BF16 activations):
  // 2^k with k = 140 - (largest E8M0), so that e2m1 * 2^(E - 127 + k) <= 6 * 2^13 for
  // the FP16-operand decode of small calls (whose GEMM takes 2^-k back on its
  // accumulators; acc_scale stays 1 for the BF16 decode).  1 for the other formats.
  float w_prescale;
  // INT4 with BF16 scales: the largest |scale| of the tensor as BF16 magnitude bits; MXFP4:
  // the largest E8M0 exponent (the repack's reduction; k is derived from it).
  int32_t max_scale_bits;
};
static_assert(sizeof(PackedHeader) <= kHeaderBytes, "header too large");

struct Layout {
  int32_t wfmt, sdtype, group, has_zp, afmt;
  int32_t groups_per_record;  // G
  int32_t scale_bytes;        // S
  int32_t record_bytes;
  int32_t off_scales, off_zeros;   // byte offsets inside a record
  int64_t N, K, N_pad, K_pad;
  int64_t n_tiles, k_blocks;
  int64_t total_bytes;
};

inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// Fills `L` from descriptor fields; returns false for unsupported combinations.
inline bool make_layout(int32_t wfmt, int32_t sdtype, int32_t group, int32_t has_zp, int32_t afmt,
                        int64_t N, int64_t K, Layout* L) {
  if (N < 1 || K < 32 || (K % 32) != 0 || N > (int64_t(1) << 31) || K > (int64_t(1) << 30))
    return false;
  if (afmt != A_BF16 && afmt != A_FP8 && afmt != A_MXFP4 && afmt != A_FP8N) return false;
  if ((afmt == A_MXFP4 || afmt == A_FP8N) && wfmt != W_MXFP4) return false;   // e2m1 operands
  if (wfmt == W_MXFP4) {
    if (sdtype != 1 || group != 32 || has_zp != 0) return false;
  } else if (wfmt == W_MXINT4 || wfmt == W_NVFP4) {
    // BF16 activations only
    if (wfmt == W_MXINT4 && (sdtype != 1 || group != 32)) return false;
    if (wfmt == W_NVFP4 && (sdtype != 2 || group != 16)) return false;
    if (has_zp != 0 || afmt != A_BF16) return false;
  } else if (wfmt == W_INT4_SYM || wfmt == W_UINT4_ZP) {
    if (sdtype != 0 || has_zp != (wfmt == W_UINT4_ZP ? 1 : 0)) return false;
    if (!(group == 32 || (group >= 64 && group % 64 == 0))) return false;
    if (afmt == A_FP8 || afmt == A_FP8N) return false;   // FP8 activations: MXFP4 weights only
  } else {
    return false;
  }
  if (K % group) return false;
  L->wfmt = wfmt; L->sdtype = sdtype; L->group = group; L->has_zp = has_zp; L->afmt = afmt;
  L->N = N; L->K = K;
  L->N_pad = round_up(N, kTileN);
  L->K_pad = round_up(K, kStageK);
  L->n_tiles = L->N_pad / kTileN;
  L->k_blocks = L->K_pad / kStageK;
  L->groups_per_record = group >= kStageK ? 1 : kStageK / group;
  L->scale_bytes = sdtype == 0 ? 2 : 1;
  L->off_scales = kCodeBytes;
  L->off_zeros = kCodeBytes + kTileN * L->groups_per_record * L->scale_bytes;
  L->record_bytes = int32_t(round_up(L->off_zeros + (has_zp ? kTileN * L->groups_per_record / 2 : 0), 16));
  L->total_bytes = round_up(kHeaderBytes + L->n_tiles * L->k_blocks * L->record_bytes, 256);
  return true;
}

// Layouts whose GEMM runs on FP16 tensor-core operands: INT4 weights with BF16 group scales
// (any group size) and BF16 activations.  A BF16 operand would round every dequantized
// weight (q - z) * s, which needs up to 12 significant bits, to 8; FP16 keeps 11.  The
// activations are then converted to FP16 exactly, with a power-of-two scale per row, by a
// pre-pass into the workspace (prep_x_f16).
inline bool f16_operands(const Layout& L) {
  return L.afmt == A_BF16 && (L.wfmt == W_INT4_SYM || L.wfmt == W_UINT4_ZP);
}

// MXFP4 and NVFP4 weights with BF16 activations: calls with token tiles of up to 64 rows
// (dense and MoE) whose workspace also holds the FP16 activation copy run on FP16
// operands, the weights decoded by the hardware e2m1x2 -> f16x2 conversion (twice the rate
// of the BF16 bit construction, where the narrow tiles make the decode the limit); wider
// tiles keep BF16 operands and need no pre-pass.  NVFP4 is exact in FP16 (e2m1 * E4M3 *
// 16 has at most 6 significant bits and stays in FP16's normal range); MXFP4 is exact like
// the BF16 decode for blocks with E >= max E - 36, blocks further below the tensor's
// largest scale falling under FP16's subnormal grid.
constexpr int kMxF16MaxTile = 64;
inline __host__ __device__ bool mx_f16_capable(const Layout& L) {
  return (L.wfmt == W_MXFP4 || L.wfmt == W_NVFP4) && L.afmt == A_BF16;
}

// Workspace bytes of the FP16 activation copy of `rows` rows: the FP16 rows [rows][K] and
// the FP32 row scales [rows], each rounded up to 256 bytes.
inline int64_t prep_x_f16_bytes(int64_t rows, int64_t K) {
  return round_up(rows * K * 2, 256) + round_up(rows * 4, 256);
}

// Device-side status codes (mirror qgemm_status values).
constexpr int kStatusBadPacked = 5;
constexpr int kStatusTimeout = 7;
constexpr int kStatusBadValue = 9;

}  // namespace qgemm
