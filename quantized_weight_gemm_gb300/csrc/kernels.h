// Host-side declarations of the kernel launchers (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qgemm_internal.h"

namespace qgemm {

int* device_status_ptr();

cudaError_t launch_repack(const Layout& L, const uint8_t* codes, const void* scales,
                          const uint8_t* zeros, void* packed, cudaStream_t st);
cudaError_t launch_dequant_debug(const Layout& L, const void* packed, void* W, cudaStream_t st);
cudaError_t launch_quant_act_fp8(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                 int64_t ldq, float* s, cudaStream_t st);

// Arguments of the tensor-core GEMM kernel (dense and MoE grouped).
struct GemmArgs {
  Layout L;                    // packed layout of one weight matrix
  const uint8_t* packed;       // expert 0
  int64_t expert_stride;       // bytes between experts (MoE), 0 for dense
  const int32_t* offsets;      // MoE: device int32 [E+1]; nullptr for dense
  int32_t E;
  int64_t M;                   // dense rows (M) or MoE rows (R)
  int32_t m_tiles, splits, num_units;   // dense schedule
  int32_t group_m;             // dense: token tiles per rasterization group (>= 1)
  const float* chan_scale;     // [N] or nullptr
  const float* tok_scale;      // [M] (FP8 activations) or nullptr
  void* Y;                     // bf16 [M, ldy]
  int64_t ldy;
  float* ws;                   // split-K partial sums [splits][m_tiles * tile_m][ws_ld]
  int32_t* counters;           // split-K arrival counters [m_tiles * n_tiles]
  int64_t ws_ld;
  int64_t ws_slice;            // floats per split slice of ws
  int* status;
  uint64_t timeout_ns;
  int32_t x_3d;                // X map is 3-D (a box covers several stages); else 2-D
};

struct GemmPlan {
  int token_tile;              // MMA N: 16, 32, 64, 128 or 256 rows of X per tile
  int splits;                  // split-K factor (dense)
  int grid;                    // persistent CTAs
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
