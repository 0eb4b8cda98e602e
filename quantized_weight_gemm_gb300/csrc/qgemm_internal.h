// Internal definitions shared by the host dispatcher and the sm_103a kernels.
//
// Packed weight layout (one weight matrix; an MoE layer stacks E of them).  The repack
// pads N to a multiple of 128 (one tile of weight rows, the M side of the tensor-core
// instruction) and K to a multiple of the stage depth BK (64 K-elements for BF16
// activations, 128 for FP8 activations), then stores:
//
//   [header: 256 B]
//   codes  : [n_tiles][k_blocks][2 or 4 chunks][128 rows][16 B]
//            chunk c of row r holds K-elements kb*BK + 32c .. +31 of that row as four
//            32-bit words of 8 nibbles; within a word the nibbles are interleaved so that
//            one mask yields two decoded lanes (see dequant.cuh).
//   scales : [n_tiles][scale_tiles_per_n][128 rows][G] entries of S bytes, where
//            G = max(1, BK / group) groups per tile, S = 2 (BF16) or 1 (E8M0).
//            For group >= BK one tile is one group and serves group/BK consecutive stages.
//   zeros  : (INT4 with zero points only) [n_tiles][scale_tiles_per_n][128 rows x G nibbles]
//            packed two rows per byte when G == 1 (row r in nibble r & 1 of byte r / 2),
//            one row per byte when G == 2 (group j of the row in nibble j).
//
// Every section starts on a 256-byte boundary and every tile is a multiple of 16 bytes,
// so each tile is one bulk asynchronous copy.
#pragma once

#include <stdint.h>

namespace qgemm {

constexpr uint32_t kPackedMagic = 0x31575147u;   // "GQW1"
constexpr uint32_t kPackedVersion = 1;
constexpr int kTileN = 128;                      // weight rows per tile (MMA M)
constexpr int kHeaderBytes = 256;

enum WFmt : int32_t { W_INT4_SYM = 0, W_UINT4_ZP = 1, W_MXFP4 = 2 };
enum AFmt : int32_t { A_BF16 = 0, A_FP8 = 1 };

struct PackedHeader {
  uint32_t magic;
  uint32_t version;
  int32_t wfmt, sdtype, group, has_zp, afmt, bk;
  int64_t N, K;
  int64_t n_tiles, k_blocks, scale_tiles;   // scale tiles per n-tile
  int64_t code_tile_bytes, scale_tile_bytes, zero_tile_bytes;
  int64_t off_codes, off_scales, off_zeros, total_bytes;
};
static_assert(sizeof(PackedHeader) <= kHeaderBytes, "header too large");

struct Layout {
  int32_t wfmt, sdtype, group, has_zp, afmt;
  int32_t bk;                 // K elements per pipeline stage
  int64_t N, K, N_pad, K_pad;
  int64_t n_tiles, k_blocks;
  int32_t groups_per_tile;    // G
  int32_t scale_bytes;        // S
  int64_t scale_tiles;        // per n-tile
  int64_t code_tile_bytes, scale_tile_bytes, zero_tile_bytes;
  int64_t off_codes, off_scales, off_zeros, total_bytes;
};

inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// Fills `L` from descriptor fields; returns false for unsupported combinations.
inline bool make_layout(int32_t wfmt, int32_t sdtype, int32_t group, int32_t has_zp, int32_t afmt,
                        int64_t N, int64_t K, Layout* L) {
  if (N < 1 || K < 32 || (K % 32) != 0 || N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
    return false;
  if (afmt != A_BF16 && afmt != A_FP8) return false;
  if (wfmt == W_MXFP4) {
    if (sdtype != 1 || group != 32 || has_zp != 0) return false;
  } else if (wfmt == W_INT4_SYM || wfmt == W_UINT4_ZP) {
    if (sdtype != 0 || has_zp != (wfmt == W_UINT4_ZP ? 1 : 0)) return false;
    if (!(group == 32 || (group >= 64 && group % 64 == 0))) return false;
    if (afmt == A_FP8) return false;    // FP8 activations pair with MXFP4 weights only
  } else {
    return false;
  }
  if (K % group) return false;
  L->wfmt = wfmt; L->sdtype = sdtype; L->group = group; L->has_zp = has_zp; L->afmt = afmt;
  L->bk = (afmt == A_FP8) ? 128 : 64;
  L->N = N; L->K = K;
  L->N_pad = round_up(N, kTileN);
  L->K_pad = round_up(K, L->bk);
  L->n_tiles = L->N_pad / kTileN;
  L->k_blocks = L->K_pad / L->bk;
  L->groups_per_tile = group >= L->bk ? 1 : L->bk / group;
  L->scale_bytes = sdtype == 0 ? 2 : 1;
  const int64_t span = group >= L->bk ? group : L->bk;       // K covered by one scale tile
  L->scale_tiles = (L->K_pad + span - 1) / span;
  L->code_tile_bytes = int64_t(kTileN) * L->bk / 2;
  L->scale_tile_bytes = int64_t(kTileN) * L->groups_per_tile * L->scale_bytes;
  L->zero_tile_bytes = has_zp ? int64_t(kTileN) * L->groups_per_tile / 2 : 0;
  L->off_codes = kHeaderBytes;
  L->off_scales = round_up(L->off_codes + L->n_tiles * L->k_blocks * L->code_tile_bytes, 256);
  L->off_zeros = round_up(L->off_scales + L->n_tiles * L->scale_tiles * L->scale_tile_bytes, 256);
  L->total_bytes = round_up(L->off_zeros + L->n_tiles * L->scale_tiles * L->zero_tile_bytes, 256);
  return true;
}

// Device-side status codes (mirror qgemm_status values).
constexpr int kStatusBadPacked = 5;
constexpr int kStatusTimeout = 7;
constexpr int kStatusBadValue = 9;

}  // namespace qgemm
