// Offline repack, dequant-debug and tokenwise FP8 activation quantization kernels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "dequant.cuh"
#include "kernels.h"
#include "qgemm_internal.h"

namespace qgemm {

__device__ int g_status = 0;

__device__ __forceinline__ void set_status(int code) { atomicCAS(&g_status, 0, code); }

int* device_status_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

// ------------------------------------------------------------------------------ repack
__device__ __forceinline__ uint8_t* record_ptr(const Layout& L, uint8_t* packed, int64_t nt,
                                               int64_t kb) {
  return packed + kHeaderBytes + (nt * L.k_blocks + kb) * int64_t(L.record_bytes);
}

// One thread writes one 16-byte chunk-row (four words) of one record's codes.
__global__ void repack_codes_kernel(Layout L, const uint8_t* __restrict__ codes,
                                    uint8_t* __restrict__ packed) {
  const int64_t total = L.n_tiles * L.k_blocks * 4 * kTileN;
  const int64_t Kh = L.K / 2;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int r = int(idx % kTileN);
    int64_t t = idx / kTileN;
    const int c = int(t % 4);
    t /= 4;
    const int64_t kb = t % L.k_blocks;
    const int64_t nt = t / L.k_blocks;
    const int64_t n = nt * kTileN + r;
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t k0 = kb * kStageK + c * 32 + j * 8;
      uint32_t src = 0;
      const bool pad = (n >= L.N) || (k0 >= L.K);
      if (!pad) src = *reinterpret_cast<const uint32_t*>(codes + n * Kh + k0 / 2);
      uint32_t w = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        uint32_t nib = pad ? 0u : (src >> (4 * e)) & 0xFu;   // even k in the low nibble
        if (L.wfmt == W_INT4_SYM || L.wfmt == W_MXINT4) nib ^= 8u;   // two's complement -> q + 8
        // natural order: the MMA's own (W4A4, FP4 operands) or the hardware e2m1x2
        // conversion's input (MXFP4 with BF16 activations)
        const bool natural = L.afmt == A_MXFP4 || L.afmt == A_FP8N || mx_f16_capable(L);
        const int pos = L.afmt == A_FP8 ? nibble_pos_a8(e) : natural ? e : nibble_pos_a16(e);
        w |= nib << (4 * pos);
      }
      out[j] = w;
    }
    uint8_t* dst = record_ptr(L, packed, nt, kb) + code_piece_offset(L.afmt, r, c);
    *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// Group of scale entry j of a record: G > 1 splits the record's 128 K into G groups; with
// G == 1 the record lies inside one group (which may span several records).
__device__ __forceinline__ int64_t record_group(const Layout& L, int64_t kb, int j) {
  return L.groups_per_record > 1 ? kb * L.groups_per_record + j : (kb * kStageK) / L.group;
}

// One thread per scale entry.
__global__ void repack_scales_kernel(Layout L, const void* __restrict__ scales,
                                     uint8_t* __restrict__ packed) {
  const int G = L.groups_per_record;
  const int64_t ngroups = L.K / L.group;
  const int64_t total = L.n_tiles * L.k_blocks * kTileN * G;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int j = int(idx % G);
    int64_t t = idx / G;
    const int r = int(t % kTileN);
    t /= kTileN;
    const int64_t kb = t % L.k_blocks;
    const int64_t nt = t / L.k_blocks;
    const int64_t n = nt * kTileN + r;
    const int64_t grp = record_group(L, kb, j);
    const bool valid = n < L.N && grp < ngroups;
    uint8_t* dst = record_ptr(L, packed, nt, kb) + L.off_scales;
    if (L.sdtype == 0) {
      uint16_t v = 0;
      if (valid) {
        v = static_cast<const uint16_t*>(scales)[n * ngroups + grp];
        if ((v & 0x7F80u) == 0x7F80u) set_status(kStatusBadValue);   // NaN / Inf
      }
      reinterpret_cast<uint16_t*>(dst)[r * G + j] = v;
      // the tensor's largest |scale| (magnitude bits order like the values): one atomic
      // per warp
      const unsigned act = __activemask();
      const int m = __reduce_max_sync(act, valid ? int(v & 0x7FFFu) : 0);
      if (int(threadIdx.x & 31) == __ffs(act) - 1)
        atomicMax(&reinterpret_cast<PackedHeader*>(packed)->max_scale_bits, m);
    } else if (L.sdtype == 1) {
      uint8_t v = 127;                                                 // E8M0 1.0
      if (valid) {
        v = static_cast<const uint8_t*>(scales)[n * ngroups + grp];
        if (v == 255) set_status(kStatusBadValue);
      }
      dst[r * G + j] = v;
      if (L.wfmt == W_MXFP4 && mx_f16_capable(L)) {   // the largest exponent, one atomic per warp
        const unsigned act = __activemask();
        const int m = __reduce_max_sync(act, valid ? int(v) : 0);
        if (int(threadIdx.x & 31) == __ffs(act) - 1)
          atomicMax(&reinterpret_cast<PackedHeader*>(packed)->max_scale_bits, m);
      }
    } else {
      uint8_t v = 0x38;                                                // E4M3 1.0
      if (valid) {
        v = static_cast<const uint8_t*>(scales)[n * ngroups + grp];
        if ((v & 0x7Fu) == 0x7Fu) set_status(kStatusBadValue);       // NaN
      }
      dst[r * G + j] = v;
    }
  }
}

// One thread per zero-point byte (two entries).
__global__ void repack_zeros_kernel(Layout L, const uint8_t* __restrict__ zeros,
                                    uint8_t* __restrict__ packed) {
  const int G = L.groups_per_record;
  const int64_t ngroups = L.K / L.group;
  const int bytes_per_rec = kTileN * G / 2;
  const int64_t total = L.n_tiles * L.k_blocks * bytes_per_rec;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int b = int(idx % bytes_per_rec);
    const int64_t t = idx / bytes_per_rec;
    const int64_t kb = t % L.k_blocks;
    const int64_t nt = t / L.k_blocks;
    uint8_t byte = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = 2 * b + h;               // entry r * G + j
      const int r = e / G, j = e % G;
      const int64_t n = nt * kTileN + r;
      const int64_t grp = record_group(L, kb, j);
      uint8_t z = 0;
      if (n < L.N && grp < ngroups) {
        z = zeros[n * ngroups + grp];
        if (z > 15) { set_status(kStatusBadValue); z &= 15; }
      }
      byte |= uint8_t(z << (4 * h));
    }
    record_ptr(L, packed, nt, kb)[L.off_zeros + b] = byte;
  }
}

__global__ void write_header_kernel(Layout L, float acc_scale, uint8_t* packed) {
  PackedHeader h;
  h.magic = kPackedMagic;
  h.version = kPackedVersion;
  h.wfmt = L.wfmt; h.sdtype = L.sdtype; h.group = L.group; h.has_zp = L.has_zp;
  h.afmt = L.afmt; h.groups_per_record = L.groups_per_record;
  h.N = L.N; h.K = L.K;
  h.n_tiles = L.n_tiles; h.k_blocks = L.k_blocks; h.record_bytes = L.record_bytes;
  h.off_scales = L.off_scales; h.off_zeros = L.off_zeros; h.total_bytes = L.total_bytes;
  h.acc_scale = acc_scale;
  h.w_prescale = 1.0f;
  h.max_scale_bits = 0;
  *reinterpret_cast<PackedHeader*>(packed) = h;
}

// FP16-operand layouts, after the scales: k = 11 - floor(log2 max|s|), clamped to
// [-100, 100], so that max|s| 2^k lies in [2^11, 2^12) and |q - z| s 2^k <= 15 * 2^12 stays
// below FP16's largest finite value; the GEMM takes 2^-k back on its accumulators.
__global__ void finish_header_f16_kernel(uint8_t* packed) {
  PackedHeader* h = reinterpret_cast<PackedHeader*>(packed);
  const int bits = h->max_scale_bits;
  int k = 0;
  if (bits != 0) {
    const int e = (bits >> 7) & 0xFF;                 // biased BF16 exponent (0: subnormal)
    int lg = e - 127;                                 // floor(log2 max|s|) for a normal
    if (e == 0) lg = -127 - (__clz(bits & 0x7F) - 25);   // subnormal: the top mantissa bit
    k = 11 - lg;
  }
  k = max(-100, min(100, k));
  h->w_prescale = ldexpf(1.0f, k);
  h->acc_scale = ldexpf(1.0f, -k);
}

// MXFP4 with BF16 activations, after the scales: k = 140 - (largest E8M0), clamped to
// [-126, 126], so that e2m1 * 2^(E - 127 + k) <= 6 * 2^13 (FP16's range) for every block;
// blocks down to 36 exponents below the largest stay exact in FP16.  The BF16 decode does
// not use it (acc_scale stays 1); the FP16-operand GEMM takes 2^-k back itself.
__global__ void finish_header_mxfp4_kernel(uint8_t* packed) {
  PackedHeader* h = reinterpret_cast<PackedHeader*>(packed);
  const int k = max(-126, min(126, 140 - h->max_scale_bits));
  h->w_prescale = ldexpf(1.0f, k);
}

static int grid_for(int64_t n) {
  const int64_t b = (n + 255) / 256;
  return int(b < 65536 ? (b > 0 ? b : 1) : 65536);
}

cudaError_t launch_repack(const Layout& L, const uint8_t* codes, const void* scales,
                          const uint8_t* zeros, float acc_scale, void* packed, cudaStream_t st) {
  uint8_t* p = static_cast<uint8_t*>(packed);
  write_header_kernel<<<1, 1, 0, st>>>(L, acc_scale, p);
  repack_codes_kernel<<<grid_for(L.n_tiles * L.k_blocks * 4 * kTileN), 256, 0, st>>>(L, codes, p);
  repack_scales_kernel<<<grid_for(L.n_tiles * L.k_blocks * kTileN * L.groups_per_record), 256, 0,
                         st>>>(L, scales, p);
  if (L.has_zp)
    repack_zeros_kernel<<<grid_for(L.n_tiles * L.k_blocks * kTileN * L.groups_per_record / 2),
                          256, 0, st>>>(L, zeros, p);
  if (f16_operands(L)) finish_header_f16_kernel<<<1, 1, 0, st>>>(p);
  if (L.wfmt == W_MXFP4 && mx_f16_capable(L)) finish_header_mxfp4_kernel<<<1, 1, 0, st>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ header check
__device__ bool header_matches(const uint8_t* packed, const Layout& L) {
  const PackedHeader* h = reinterpret_cast<const PackedHeader*>(packed);
  return h->magic == kPackedMagic && h->version == kPackedVersion && h->wfmt == L.wfmt &&
         h->sdtype == L.sdtype && h->group == L.group && h->has_zp == L.has_zp &&
         h->afmt == L.afmt && h->N == L.N && h->K == L.K && h->total_bytes == L.total_bytes;
}

// ------------------------------------------------------------------------ dequant debug
// One thread decodes one packed word (8 K-elements of one row) through the GEMM decoders.
__global__ void dequant_debug_kernel(Layout L, const uint8_t* __restrict__ packed,
                                     __nv_bfloat16* __restrict__ W) {
  __shared__ int ok;
  if (threadIdx.x == 0) {
    ok = header_matches(packed, L);
    if (!ok && blockIdx.x == 0) set_status(kStatusBadPacked);
  }
  __syncthreads();
  if (!ok) return;
  const int64_t total = L.n_tiles * L.k_blocks * 4 * kTileN * 4;
  const int G = L.groups_per_record;
  for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < total;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int j = int(idx % 4);
    int64_t t = idx / 4;
    const int r = int(t % kTileN);
    t /= kTileN;
    const int c = int(t % 4);
    t /= 4;
    const int64_t kb = t % L.k_blocks;
    const int64_t nt = t / L.k_blocks;
    const int64_t n = nt * kTileN + r;
    const int64_t k0 = kb * kStageK + c * 32 + j * 8;
    if (n >= L.N || k0 >= L.K) continue;
    const uint8_t* rec = packed + kHeaderBytes + (nt * L.k_blocks + kb) * int64_t(L.record_bytes);
    const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + code_piece_offset(L.afmt, r, c) + j * 4);
    const int js = c * G / 4;                          // scale entry of chunk c
    const int ent = r * G + js;
    __nv_bfloat16* dst = W + n * L.K + k0;
    if (L.afmt == A_MXFP4 || L.afmt == A_FP8N) {
      // the MMA's operand: e2m1 codes in natural order, times 2^(E-127) (exact in bf16)
      const uint32_t E = rec[L.off_scales + ent];
      for (int e = 0; e < 8; ++e) {
        const uint32_t q = (w >> (4 * e)) & 0xFu;
        const uint32_t mag = q & 7u;
        float v = mag < 2 ? 0.5f * float(mag) : ldexpf(1.0f + 0.5f * float(mag & 1u), int(mag >> 1) - 1);
        v = ldexpf(v, int(E) - 127);
        dst[e] = __float2bfloat16_rn((q & 8u) ? -v : v);
      }
      continue;
    }
    if (L.afmt == A_FP8) {
      // e2m1 -> e4m3 byte shuffle, then value = e4m3 * 2^6 * 2^(E-127) (exact in bf16)
      const uint32_t E = rec[L.off_scales + ent];
      uint32_t lo, hi;
      decode_e2m1_to_e4m3_word(w, lo, hi);
      for (int e = 0; e < 8; ++e) {
        const uint32_t b = ((e < 4 ? lo : hi) >> (8 * (e & 3))) & 0xFFu;
        const uint32_t ex = (b >> 3) & 0xFu, m = b & 7u;
        float v = ex == 0 ? ldexpf(float(m) / 8.0f, -6) : ldexpf(1.0f + float(m) / 8.0f, int(ex) - 7);
        v = ldexpf(v, 6 + int(E) - 127);
        if (b & 0x80u) v = -v;
        dst[e] = __float2bfloat16_rn(v);
      }
      continue;
    }
    uint32_t out[4];
    if (L.wfmt == W_NVFP4) {
      // the GEMM's decode (e2m1 x s x 2^-8, exact), then the accumulator factor (2^8 times
      // the per-tensor scale) in double and one rounding to BF16
      const uint32_t s = e4m3_bf16x2_p118(rec[L.off_scales + r * G + c * 2 + j / 2]);
      decode_mxfp4_word_nat(w, s, 0u, false, out);
      const double f = double(reinterpret_cast<const PackedHeader*>(packed)->acc_scale);
      for (int e = 0; e < 8; ++e) {
        const uint32_t hb = (out[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
        dst[e] = __double2bfloat16(double(__uint_as_float(hb << 16)) * f);
      }
      continue;
    }
    if (L.wfmt == W_MXFP4) {
      const uint32_t E = rec[L.off_scales + ent];
      uint32_t sa, sb;
      bool big;
      mxfp4_factors(E, sa, sb, big);
      decode_mxfp4_word_nat(w, sa, sb, big, out);
    } else if (L.wfmt == W_MXINT4) {
      decode_int4_word(w, 0x43084308u, e8m0_bf16x2(rec[L.off_scales + ent]), out);
    } else {
      const uint32_t s = reinterpret_cast<const uint16_t*>(rec + L.off_scales)[ent];
      uint32_t z = 8;
      if (L.has_zp) z = (rec[L.off_zeros + ent / 2] >> (4 * (ent & 1))) & 0xFu;
      const uint32_t zz = (0x4300u | z) * 0x00010001u;
      decode_int4_word(w, zz, s * 0x00010001u, out);
    }
    // pair i = elements (2i, 2i+1): low half is the even element
    *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

cudaError_t launch_dequant_debug(const Layout& L, const void* packed, void* W, cudaStream_t st) {
  const int64_t total = L.n_tiles * L.k_blocks * 4 * kTileN * 4;
  dequant_debug_kernel<<<grid_for(total), 256, 0, st>>>(L, static_cast<const uint8_t*>(packed),
                                                       static_cast<__nv_bfloat16*>(W));
  return cudaGetLastError();
}

// --------------------------------------------------------- FP16 activations (pre-pass)
// One block of 256 threads per row.  A row of up to 32768 elements stays in registers
// (16-byte loads, at most 16 per thread): the maximum of |x| (BF16 magnitude bits order
// like the values), then every element times 2^-e (exact in FP32) rounded once to FP16,
// 16-byte stores.  Longer rows are read twice.  The block first lets dependent launches
// start (programmatic dependent launch): the GEMM's prologue and weight stream overlap
// this pass, and its activation reads wait for it to finish.
constexpr int kPrepThreads = 256, kPrepVecs = 16;

__device__ __forceinline__ uint32_t bf16x8_absmax(uint4 v) {
  const uint32_t a = max(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  const uint32_t b = max(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
  const uint32_t c = __vmaxu2(a, b);                  // per 16-bit half
  return max(c & 0xFFFFu, c >> 16);
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v, float inv) {
  const float lo = __uint_as_float(v << 16) * inv, hi = __uint_as_float(v & 0xFFFF0000u) * inv;
  return ptx::cvt_f16x2_f32(lo, hi);
}

__global__ void __launch_bounds__(kPrepThreads)
prep_x_f16_kernel(const uint8_t* __restrict__ X, int64_t K, int64_t ldx_bytes,
                  uint8_t* __restrict__ X16, float* __restrict__ rowscale) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t m = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(X + m * ldx_bytes);
  uint4* yr = reinterpret_cast<uint4*>(X16 + m * K * 2);
  const int nv = int(K / 8);                          // 16-byte vectors in the row
  const bool in_regs = nv <= kPrepThreads * kPrepVecs;
  uint4 v[kPrepVecs];
  uint32_t amax = 0;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kPrepVecs; ++i) {
      const int j = threadIdx.x + i * kPrepThreads;
      v[i] = j < nv ? __ldg(xr + j) : make_uint4(0, 0, 0, 0);
      amax = max(amax, bf16x8_absmax(v[i]));
    }
  } else {
    for (int j = threadIdx.x; j < nv; j += kPrepThreads) amax = max(amax, bf16x8_absmax(__ldg(xr + j)));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  __shared__ uint32_t red[kPrepThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kPrepThreads / 32; ++i) amax = max(amax, red[i]);
  int e = 0;                                          // floor(log2 amax) - 14
  const uint32_t be = (amax >> 7) & 0xFFu;
  if (amax != 0 && be != 0xFFu) {
    const int lg = be != 0 ? int(be) - 127 : -127 - (__clz(amax & 0x7Fu) - 25);
    e = lg - 14;
  }
  const float inv = ldexpf(1.0f, -e);
  auto cvt8 = [&](uint4 a) {
    return make_uint4(bf16x2_to_f16x2(a.x, inv), bf16x2_to_f16x2(a.y, inv),
                      bf16x2_to_f16x2(a.z, inv), bf16x2_to_f16x2(a.w, inv));
  };
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < kPrepVecs; ++i) {
      const int j = threadIdx.x + i * kPrepThreads;
      if (j < nv) yr[j] = cvt8(v[i]);
    }
  } else {
    for (int j = threadIdx.x; j < nv; j += kPrepThreads) yr[j] = cvt8(__ldg(xr + j));
  }
  if (threadIdx.x == 0) rowscale[m] = ldexpf(1.0f, e);
}

cudaError_t launch_prep_x_f16(const void* X, int64_t rows, int64_t K, int64_t ldx, void* X16,
                              float* rowscale, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  prep_x_f16_kernel<<<unsigned(rows), kPrepThreads, 0, st>>>(
      static_cast<const uint8_t*>(X), K, ldx * 2, static_cast<uint8_t*>(X16), rowscale);
  return cudaGetLastError();
}

// ------------------------------------------------------------ indexed MoE: row gather
// One warp per sorted position r: dst row r = src row idx[r] (row_bytes bytes, 16-byte
// vectors), or zeros for a negative index; an index past the end sets the bad-value status
// and gives zeros.  With scales, dst_scale[r] = src_scale[idx[r]] (0 for padding).
constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32)
gather_rows_kernel(const uint8_t* __restrict__ src, int64_t src_ld, int64_t src_rows,
                   const int32_t* __restrict__ idx, int64_t R, int64_t row_bytes,
                   uint8_t* __restrict__ dst, int64_t dst_ld, const float* __restrict__ src_scale,
                   float* __restrict__ dst_scale, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t r = int64_t(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5);
  if (r >= R) return;
  const int32_t t = idx[r];
  const bool ok = t >= 0 && t < src_rows;
  if (lane == 0 && t >= src_rows) atomicCAS(status, 0, kStatusBadValue);
  uint4* d = reinterpret_cast<uint4*>(dst + r * dst_ld);
  const int64_t nv = row_bytes / 16;
  if (ok) {
    const uint4* s = reinterpret_cast<const uint4*>(src + int64_t(t) * src_ld);
    int64_t v = lane;
    for (; v + 96 < nv; v += 128) {        // four 16-byte loads in flight per lane
      const uint4 a0 = __ldg(s + v), a1 = __ldg(s + v + 32), a2 = __ldg(s + v + 64),
                  a3 = __ldg(s + v + 96);
      d[v] = a0; d[v + 32] = a1; d[v + 64] = a2; d[v + 96] = a3;
    }
    for (; v < nv; v += 32) d[v] = __ldg(s + v);
  } else {
    for (int64_t v = lane; v < nv; v += 32) d[v] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (dst_scale != nullptr && lane == 0) dst_scale[r] = ok ? src_scale[t] : 0.0f;
}

cudaError_t launch_gather_rows(const void* src, int64_t src_ld, int64_t src_rows,
                               const int32_t* idx, int64_t R, int64_t row_bytes, void* dst,
                               int64_t dst_ld, const float* src_scale, float* dst_scale,
                               int* status, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  const int64_t blocks = (R + kGatherWarps - 1) / kGatherWarps;
  gather_rows_kernel<<<unsigned(blocks), kGatherWarps * 32, 0, st>>>(
      static_cast<const uint8_t*>(src), src_ld, src_rows, idx, R, row_bytes,
      static_cast<uint8_t*>(dst), dst_ld, src_scale, dst_scale, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------ MXFP4 act quantization
// One warp per 32-element block (lane = element), 8 warps per block of rows: the block's
// largest |x| (BF16 magnitude bits), E = floor(log2 amax) - 2 + 127 clamped to [0, 254]
// (127 for an all-zero block), each x * 2^(127 - E) (exact in FP32) rounded to e2m1 by the
// hardware conversion (nearest even, saturating at 6).  Codes: byte j of the block holds
// elements 2j (low nibble) and 2j + 1; blocks of a row past K (up to the exps row's
// padding to a multiple of 4) get E = 127.
__global__ void quant_act_mxfp4_kernel(const uint16_t* __restrict__ X, int64_t M, int64_t K,
                                       int64_t ldx, uint8_t* __restrict__ Xq, int64_t ldq,
                                       uint8_t* __restrict__ exps, int64_t lde, int64_t nblk_pad) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t nblk = K / 32;
  for (int64_t t = warp_global; t < M * nblk_pad; t += nwarps) {
    const int64_t m = t / nblk_pad, b = t % nblk_pad;
    if (b >= nblk) {                                   // padding block of the exps row
      if (lane == 0) exps[m * lde + b] = 127;
      continue;
    }
    const uint32_t bits = X[m * ldx + b * 32 + lane];
    const uint32_t amax = __reduce_max_sync(0xffffffffu, bits & 0x7FFFu);
    int E = 127;
    const uint32_t be = (amax >> 7) & 0xFFu;
    if (amax != 0) {
      const int lg = be != 0 ? int(be) - 127 : -127 - (__clz(amax & 0x7Fu) - 25);
      E = max(0, min(254, lg - 2 + 127));
    }
    const float v = ldexpf(__uint_as_float(bits << 16), 127 - E);
    const float hi = __shfl_down_sync(0xffffffffu, v, 1);
    uint32_t byte = ptx::cvt_e2m1x2_f32(v, hi) & 0xFFu;   // even lanes: elements 2j, 2j + 1
    // bytes of lanes 8k, 8k+2, 8k+4, 8k+6 -> one 32-bit word at lane 8k
    const uint32_t b1 = __shfl_down_sync(0xffffffffu, byte, 2);
    const uint32_t b2 = __shfl_down_sync(0xffffffffu, byte, 4);
    const uint32_t b3 = __shfl_down_sync(0xffffffffu, byte, 6);
    if ((lane & 7) == 0)
      *reinterpret_cast<uint32_t*>(Xq + m * ldq + b * 16 + (lane >> 3) * 4) =
          byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
    if (lane == 0) exps[m * lde + b] = uint8_t(E);
  }
}

cudaError_t launch_quant_act_mxfp4(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                   int64_t ldq, uint8_t* exps, int64_t lde, cudaStream_t st) {
  const int64_t nblk_pad = (K / 32 + 3) / 4 * 4;      // whole 128-K blocks (the GEMM reads words)
  const int64_t warps = M * nblk_pad;
  const int64_t blocks = std::min<int64_t>((warps + 7) / 8, 152 * 16);
  quant_act_mxfp4_kernel<<<unsigned(std::max<int64_t>(blocks, 1)), 256, 0, st>>>(
      static_cast<const uint16_t*>(X), M, K, ldx, Xq, ldq, exps, lde, nblk_pad);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ FP8 act quantization
// One block of 256 threads per row: float32 row maximum, s = amax / 448, code = e4m3
// RNE-satfinite of x / s (IEEE float32 division).
__global__ void __launch_bounds__(256) quant_act_fp8_kernel(const __nv_bfloat16* __restrict__ X,
                                                            int64_t K, int64_t ldx,
                                                            uint8_t* __restrict__ Xq, int64_t ldq,
                                                            float* __restrict__ s_out) {
  const int64_t m = blockIdx.x;
  const __nv_bfloat16* x = X + m * ldx;
  float amax = 0.0f;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(__bfloat162float(x[k])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < 8 ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  amax = red[0];
  const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
  if (threadIdx.x == 0) s_out[m] = s;
  uint8_t* q = Xq + m * ldq;
  for (int64_t k = 2 * threadIdx.x; k < K; k += 2 * blockDim.x) {
    const float a = __fdiv_rn(__bfloat162float(x[k]), s);
    const float b = (k + 1 < K) ? __fdiv_rn(__bfloat162float(x[k + 1]), s) : 0.0f;
    const uint16_t pair = ptx::cvt_e4m3x2_f32(a, b);
    q[k] = uint8_t(pair & 0xFF);
    if (k + 1 < K) q[k + 1] = uint8_t(pair >> 8);
  }
}

// The same computation on 16-byte vectors: each thread keeps its first kKeep vectors of the
// row in registers between the maximum and the quantization, later ones are read again
// (from L2).  Requires K % 8 == 0, X and every row 16-byte aligned, Xq rows 8-byte aligned.
constexpr int kQThreads = 256, kKeep = 4;

__device__ __forceinline__ float amax8(uint4 v, float a) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a = fmaxf(a, fabsf(__uint_as_float(w[i] << 16)));
    a = fmaxf(a, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
  }
  return a;
}

__device__ __forceinline__ uint2 quant8(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = ptx::cvt_e4m3x2_f32(__fdiv_rn(__uint_as_float(w[i] << 16), s),
                               __fdiv_rn(__uint_as_float(w[i] & 0xFFFF0000u), s));
  return make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
}

__global__ void __launch_bounds__(kQThreads) quant_act_fp8_vec_kernel(
    const __nv_bfloat16* __restrict__ X, int64_t K, int64_t ldx, uint8_t* __restrict__ Xq,
    int64_t ldq, float* __restrict__ s_out) {
  const int64_t m = blockIdx.x;
  const uint4* x = reinterpret_cast<const uint4*>(X + m * ldx);
  const int64_t nv = K / 8;
  uint4 keep[kKeep];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kKeep; ++i) {
    const int64_t j = int64_t(i) * kQThreads + threadIdx.x;
    keep[i] = j < nv ? __ldg(x + j) : make_uint4(0, 0, 0, 0);
    amax = amax8(keep[i], amax);
  }
  for (int64_t j = int64_t(kKeep) * kQThreads + threadIdx.x; j < nv; j += kQThreads)
    amax = amax8(__ldg(x + j), amax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[kQThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, red[i]);
  const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
  if (threadIdx.x == 0) s_out[m] = s;
  uint2* q = reinterpret_cast<uint2*>(Xq + m * ldq);
#pragma unroll
  for (int i = 0; i < kKeep; ++i) {
    const int64_t j = int64_t(i) * kQThreads + threadIdx.x;
    if (j < nv) q[j] = quant8(keep[i], s);
  }
  for (int64_t j = int64_t(kKeep) * kQThreads + threadIdx.x; j < nv; j += kQThreads)
    q[j] = quant8(__ldg(x + j), s);
}

cudaError_t launch_quant_act_fp8(const void* X, int64_t M, int64_t K, int64_t ldx, uint8_t* Xq,
                                 int64_t ldq, float* s, cudaStream_t st) {
  const bool vec = K % 8 == 0 && ldx % 8 == 0 && ldq % 8 == 0 &&
                   reinterpret_cast<uintptr_t>(X) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(Xq) % 8 == 0;
  if (vec)
    quant_act_fp8_vec_kernel<<<unsigned(M), kQThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(X), K, ldx, Xq, ldq, s);
  else
    quant_act_fp8_kernel<<<unsigned(M), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(X), K,
                                                      ldx, Xq, ldq, s);
  return cudaGetLastError();
}

}  // namespace qgemm
