// Device-side helpers shared by the kernels of the library: FP4/FP8 code
// conversion, page addressing, error reporting.  Written from the OCP MX v1.0
// (E2M1) and OCP OFP8 (E4M3, FN variant) definitions and the byte layout of
// include/pkv.h; nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/pkv.h"

#define PKV_PAGE 64
#define PKV_WINDOW 128

// device error word bits (pkv_get_error maps them to pkv_status)
#define PKV_DEVERR_BAD_PAGE 1
#define PKV_DEVERR_TIMEOUT 2

namespace pkv {

__device__ __forceinline__ void report(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------- dependent launch
// A kernel started by launch_pdl may begin while the kernel before it in the
// stream is still running (programmatic dependent launch).  Before it reads or
// writes anything in global memory it calls dep_wait(), which returns once that
// kernel has finished and its writes are visible; dep_trigger() then lets the
// next kernel of the stream start.  Called after dep_wait(), it keeps at most
// two kernels of a stream on the GPU at once.  Both are no-ops in a kernel
// launched the plain way.
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialization (the kernel must call dep_wait()
// before touching global memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------- encoders
// E4M3 code of a finite a >= 0: nearest finite value, ties to the even code,
// saturating at 448 (0x7E).  Subnormals (a < 2^-6) are multiples of 2^-9.
__device__ __forceinline__ uint32_t e4m3_code_pos(float a) {
  if (!(a < 448.f)) return 0x7Eu;
  if (a < 0.015625f) {                       // 2^-6
    return (uint32_t)__float2int_rn(a * 512.f);   // exact scaling; RNE -> 0..8 (8 = 2^-6, code 0x08)
  }
  const uint32_t u = __float_as_uint(a);
  int e = (int)(u >> 23) - 127 + 7;           // biased E4M3 exponent, >= 1
  const uint32_t m = u & 0x7FFFFFu;
  uint32_t keep = m >> 20;                    // 3 kept mantissa bits
  const uint32_t rem = m & 0xFFFFFu;          // 20 dropped bits
  keep += (rem > 0x80000u) || (rem == 0x80000u && (keep & 1u));
  if (keep == 8u) { keep = 0u; e += 1; }
  const uint32_t code = ((uint32_t)e << 3) | keep;
  return code > 0x7Eu ? 0x7Eu : code;
}

__device__ __forceinline__ uint32_t e4m3_code(float x) {
  return e4m3_code_pos(fabsf(x)) | (signbit(x) ? 0x80u : 0u);
}

// E2M1 code of v: magnitude grid {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even
// code (the grid points with even codes win their midpoints), |v| >= 6 -> 6.
__device__ __forceinline__ uint32_t e2m1_code(float v) {
  const float a = fabsf(v);
  const uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) +
                     (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
  return c | (signbit(v) ? 8u : 0u);
}

// ---------------------------------------------------------------- decoders
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  const float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
  return (c & 0x80u) ? -v : v;
}

__device__ __forceinline__ float e2m1_value(uint32_t c) {
  // magnitudes of codes 0..7 are 0, .5, 1, 1.5, 2, 3, 4, 6
  const uint32_t m = c & 7u;
  const float mag = (m < 4u) ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1u)) * ((m & 1u) ? 1.5f : 1.0f);
  return (c & 8u) ? -mag : mag;
}

// ---------------------------------------------------------------- page layout
// K cache: a token's d/2 code bytes are cut into column blocks of RB = min(128, d/2)
// bytes stored [column block][64 tokens][RB]; inside a block the 16-byte chunk c
// of token t sits at chunk position c ^ w(t), w = t mod 8 (RB = 128) or
// (t / 2) mod 4 (RB = 64): the K-major operand layout (128- / 64-byte swizzle)
// of the block-scaled FP4 contraction, so pages are consumed as copied.
template <int D>
struct KLayout {
  static constexpr int RB = D / 2 < 128 ? D / 2 : 128;
  static constexpr int CPR = RB / 16;          // 16-byte chunks per row of a column block
  __host__ __device__ static constexpr int swz(int t) { return RB == 128 ? (t & 7) : ((t >> 1) & 3); }
  // byte offset of 16-byte chunk c (channels 32c .. 32c+31) of token t
  __device__ __forceinline__ static int chunk(int t, int c) {
    return (c / CPR) * (PKV_PAGE * RB) + t * RB + 16 * ((c % CPR) ^ swz(t));
  }
  // byte offset of channel pair j (channels 2j, 2j+1) of token t
  __device__ __forceinline__ static int data(int t, int j) { return chunk(t, j >> 4) + (j & 15); }
  // byte offset of the scale of block j of token t
  __device__ __forceinline__ static int scale(int t, int j) {
    return (((j >> 3) * PKV_PAGE + t) << 3) + (j & 7);
  }
};

// Index keys (128 channels): rows of 64 bytes, 16-byte chunk c of token t at
// chunk position c ^ (t mod 4); scales as the K cache.
struct IdxLayout {
  __device__ __forceinline__ static int data(int t, int j) { return t * 64 + 16 * ((j >> 4) ^ (t & 3)) + (j & 15); }
  __device__ __forceinline__ static int scale(int t, int j) { return (((j >> 3) * PKV_PAGE + t) << 3) + (j & 7); }
};

// V cache: channel-major 32-bit words grouped by 128-channel chunk,
// [d/128 chunks][8 token octets][128 channels]: word (chunk c/128, octet t/8,
// channel c%128) holds channel c of tokens 8*(t/8) .. 8*(t/8)+7 (nibble t%8), so
// one 128-channel chunk of a page is one contiguous 4 KB run.
template <int D>
struct VLayout {
  __device__ __forceinline__ static int word(int t, int c) { return (((c >> 7) * 8 + (t >> 3)) << 7) + (c & 127); }
  __device__ __forceinline__ static int scale(int t, int j) { return j * PKV_PAGE + t; }
};

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

}  // namespace pkv
