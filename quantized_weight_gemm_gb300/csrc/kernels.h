// Host-side declarations of the kernel launchers (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qgemm.h"
#include "qgemm_internal.h"

namespace qgemm {

// The scratch that the dense W4A16 call would use for these arguments under its own plan
// for M, given at most `capacity` bytes: *need bytes in all (the FP16 activation copy where
// the call makes one -- always for INT4 with BF16 scales, for small MXFP4 calls when it fits
// the capacity -- then the partial sums of cut tiles; 0 for neither), of which the arrival
// counters, [*counter_off, *counter_off + *counter_bytes), must be zero at launch.  Checks
// every argument as qgemm_w4a16 does and returns its error, if any, before looking at the
// device.  qgemm_w4a16 given exactly *need bytes of workspace runs the same schedule.
qgemm_status dense_a16_scratch(const qgemm_wdesc* desc, const void* packed, const void* X,
                               int64_t M, int64_t ldx, const float* chan_scale, const void* Y,
                               int64_t ldy, int64_t capacity, int64_t* need,
                               int64_t* counter_off, int64_t* counter_bytes);

int* device_status_ptr();

// acc_scale: the factor the GEMM applies to its accumulators, stored in the header.
cudaError_t launch_repack(const Layout& L, const uint8_t* codes, const void* scales,
                          const uint8_t* zeros, float acc_scale, void* packed, cudaStream_t st);
cudaError_t launch_dequant_debug(const Layout& L, const void* packed, void* W, cudaStream_t st);
// The FP16 copy of BF16 activations for the FP16-operand GEMM: for each row m,
// e_m = floor(log2(amax_m)) - 14 (0 for an all-zero row), X16[m][k] = X[m][k] * 2^-e_m
// rounded to FP16 (exact unless |x| < 2^-31 amax_m, below FP16's subnormal grid),
// rowscale[m] = 2^e_m.  X16 is [rows][K] with leading dimension K.
cudaError_t launch_prep_x_f16(const void* X, int64_t rows, int64_t K, int64_t ldx, void* X16,
                              float* rowscale, cudaStream_t st);
// MXFP4 activations for W4A4: codes [M][ldq] bytes (element 2j in the low nibble of byte j)
// and E8M0 exponents [M][lde] bytes, one per 32 K, blocks past K up to a multiple of 4
// filled with 127.
cudaError_t launch_quant_act_mxfp4(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                   int64_t ldq, uint8_t* exps, int64_t lde, cudaStream_t st);
cudaError_t launch_quant_act_fp8(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                 int64_t ldq, float* s, cudaStream_t st);
// Indexed MoE: dst row r (dst_ld bytes apart) = src row idx[r] (src_ld bytes apart, src_rows
// rows), row_bytes bytes (a multiple of 16, both pointers and strides 16-byte aligned); a
// negative index gives a zero row, an index >= src_rows sets kStatusBadValue in *status and
// gives a zero row.  If dst_scale is given, dst_scale[r] = src_scale[idx[r]] (0 for padding).
cudaError_t launch_gather_rows(const void* src, int64_t src_ld, int64_t src_rows,
                               const int32_t* idx, int64_t R, int64_t row_bytes, void* dst,
                               int64_t dst_ld, const float* src_scale, float* dst_scale,
                               int* status, cudaStream_t st);

// Arguments of the tensor-core GEMM kernel (dense and MoE grouped).
struct GemmArgs {
  Layout L;                    // packed layout of one weight matrix
  const uint8_t* packed;       // expert 0
  int64_t expert_stride;       // bytes between experts (MoE), 0 for dense
  const int32_t* offsets;      // MoE: device int32 [E+1]; nullptr for dense
  // Indexed MoE: device int32 [R], the X row of sorted position r (negative: padding);
  // nullptr otherwise.  The gathering kernel copies those rows from x itself (no tensor map).
  const int32_t* row_index;
  const uint8_t* x;            // indexed MoE: X in token order, x_rows rows of ldx_bytes
  int64_t ldx_bytes;
  int64_t x_rows;
  int32_t E;
  int64_t M;                   // dense rows (M) or MoE rows (R)
  // Dense schedule.  Tiles are numbered in rasterization order (groups of group_m token
  // tiles, the token tile changing fastest inside a group).
  //  - sk_tiles == 0: units = (tile, split) pairs, unit u on CTA u % grid; splits == 1 is
  //    plain data-parallel, splits > 1 cuts every tile's K range into `splits` equal parts.
  //  - sk_tiles > 0 ("stream-K"): the records of tiles [0, sk_tiles) are dealt out evenly
  //    as contiguous ranges, CTA i taking records [i S / grid, (i + 1) S / grid) of the
  //    S = sk_tiles * k_blocks; after its range a CTA takes the whole tiles
  //    sk_tiles + i, sk_tiles + i + grid, ...  (MoE: decided in the kernel.)
  int32_t m_tiles, splits, num_units;
  int32_t group_m;             // token tiles per rasterization group (>= 1)
  int32_t sk_tiles;
  const float* chan_scale;     // [N] or nullptr
  // Bias added after every scale: [N] (dense, bias_stride 0) or [E][N] (MoE, bias_stride N),
  // or nullptr.
  const float* bias;
  int64_t bias_stride;
  const float* tok_scale;      // [M] (FP8 activations) or nullptr
  // MXFP4 activations (W4A4): E8M0 exponents, row m at x_exps + m * ld_exps bytes, one
  // 32-bit word (four exponents) per 128-K block; tmap_e describes them for TMA as a 2-D
  // uint8 tensor [rows][ld_exps] loaded in boxes of 16 bytes (four blocks) x token_tile rows
  const uint8_t* x_exps;
  int64_t ld_exps;
  CUtensorMap tmap_e;
  // FP8 activations on FP4 operands (afmt A_FP8N): the packed codes as a 4-D tensor
  // [experts][records][128 rows][128 e2m1] (strides expert_stride, record_bytes, 64 bytes),
  // loaded one record at a time into the padded 128-byte rows the MMA reads
  CUtensorMap tmap_w;
  void* Y;                     // bf16 [M, ldy]
  int64_t ldy;
  // Partial sums of the tiles whose K range is cut over several CTAs: one slot per
  // contributor, an FP32 tile [128 weight rows][token_tile], row-major (uniform cuts: slot
  // tile * splits + split; stream-K: slot t + first(t) + j, fewer than sk_tiles + grid, or
  // with fewer records S than CTAs the record's own index, below S).
  // MoE: optional; when given, the kernel may run stream-K (2 * grid slots).
  float* ws;
  int32_t* counters;           // arrival counter per cut tile (zero between calls)
  int* status;
  uint64_t timeout_ns;
  int32_t x_3d;                // X map is 3-D (a box covers several stages); else 2-D
  // Test aid (qgemm_debug_stall): the activation producer of each CTA never issues its
  // first load, so the waits on it run into their time limit; nothing is left in flight.
  int32_t debug_skip_first_x;
};

struct GemmPlan {
  int token_tile;              // MMA N: 16, 32, 64, 128 or 256 rows of X per tile
  int splits;                  // split-K factor (dense, uniform cut; 1 = none)
  int sk_tiles;                // > 0: stream-K over the first sk_tiles tiles (splits == 1)
  int max_contrib;             // partial-sum slots per cut tile (0 when nothing is cut)
  int grid;                    // persistent CTAs
  // Launched as a programmatic dependent of the kernel before it on the stream (the FP16
  // activation pre-pass): its prologue and weight stream start early, and its reads of the
  // pre-pass's output wait for that kernel (griddepcontrol.wait).
  int pdl = 0;
  // MXFP4 weights with BF16 activations: FP16 operands (the activation copy made by the
  // pre-pass, the weights decoded by the hardware e2m1 conversion); see mx_f16_capable().
  int mx_f16 = 0;
};

// Launch the tcgen05 GEMM for the given plan.  tmap describes X (BF16 or E4M3, K-major,
// 128-byte swizzle): either 2-D with box {one 128-byte slab, token_tile rows}, or (args.x_3d)
// 3-D [K / slab][rows][slab] with box {slab, token_tile, gemm_x_box_slabs()}.
cudaError_t launch_gemm(bool fp8, const GemmPlan& plan, const CUtensorMap& tmap,
                        const GemmArgs& args, cudaStream_t st);

// Dynamic shared memory bytes of a variant (for occupancy checks / attributes).
int gemm_smem_bytes(bool fp8, int token_tile);

// Number of 128-byte X slabs one 3-D activation load covers (several stages' worth for
// narrow token tiles, one stage otherwise).
int gemm_x_box_slabs(bool fp8, int token_tile);

}  // namespace qgemm
