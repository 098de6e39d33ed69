// pair_tile.cuh -- building blocks of the per-pair tensor-core kernels (backward pass, triangle
// attention): 128 x 128 bf16 operand tiles in the 128-byte-swizzled K-major layout that one CTA's
// threads fill row by row, their tcgen05 descriptors read K-major (K = the tile's columns) or
// MN-major (K = the tile's rows), and small register helpers.
#pragma once
#include "tm_kernels.h"

namespace tmk {
namespace pt {

constexpr int BT = 128;                 // pairs per tile
constexpr int NT = 512;                 // threads per CTA: 4 per pair, 32 channels each
constexpr uint32_t TILE = 128 * 128 * 2;  // bytes of one 128 x 128 bf16 operand tile
constexpr uint32_t SLAB = TILE / 2;       // one 64-channel half


// 8 floats -> one 16-byte unit of row `r` of an operand tile, for channels c0 .. c0+7 (c0 % 8 == 0),
// as bf16 (put8) or fp16 (put8h)
__device__ __forceinline__ void put8(uint8_t* tile, int r, int c0, const float* v) {
  const uint4 q = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                             pack_bf16x2(v[6], v[7]));
  *reinterpret_cast<uint4*>(tile + (c0 >> 6) * SLAB + sw128_offset((uint32_t)r, (uint32_t)((c0 & 63) >> 3))) = q;
}
__device__ __forceinline__ void put8h(uint8_t* tile, int r, int c0, const float* v) {
  const uint4 q = make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                             pack_f16x2(v[6], v[7]));
  *reinterpret_cast<uint4*>(tile + (c0 >> 6) * SLAB + sw128_offset((uint32_t)r, (uint32_t)((c0 & 63) >> 3))) = q;
}

__device__ __forceinline__ void f16x8_to_float(const uint4& q, float* f) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
    f[2 * k] = t.x;
    f[2 * k + 1] = t.y;
  }
}

// 8 floats as fp16 in one 16-byte word
__device__ __forceinline__ uint4 pack8h(const float* v) {
  return make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]), pack_f16x2(v[6], v[7]));
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& q, float* f) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

// Copy a weight image (already in the tile layout, 16-bit elements) into shared memory, all threads.
__device__ __forceinline__ void copy_tile(uint8_t* dst, const void* src) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll 4
  for (int k = threadIdx.x; k < (int)(TILE / 16); k += NT) d[k] = s[k];
}

// 32 bf16 values (64 bytes) -> floats
__device__ __forceinline__ void load32_bf16(const __nv_bfloat16* src, float* f) {
  const uint4* q = reinterpret_cast<const uint4*>(src);
  uint4 v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) v[u] = q[u];
#pragma unroll
  for (int u = 0; u < 4; ++u) bf16x8_to_float(v[u], f + 8 * u);
}

// 32 fp16 values (64 bytes) -> floats
__device__ __forceinline__ void load32_f16(const __half* src, float* f) {
  const uint4* q = reinterpret_cast<const uint4*>(src);
  uint4 v[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) v[u] = q[u];
#pragma unroll
  for (int u = 0; u < 4; ++u) f16x8_to_float(v[u], f + 8 * u);
}

// Butterfly reduce-scatter over the 32 lanes of a warp: on return lane l holds the sum over the
// lanes of v[l] (v is consumed).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float keep = upper ? v[k + half] : v[k];
      const float send = upper ? v[k] : v[k + half];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  return v[0];
}

// Issue helpers (one thread). K-major operand of a 128 x 128 tile: K = channels; MN-major operand:
// K = the tile's rows (pairs, or the out index of a weight image).
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int ks) {
  return make_sdesc_sw128(base + (uint32_t)((ks >> 2) * SLAB + (ks & 3) * 32), 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc(uint32_t base, int ks) {
  return make_sdesc_sw128(base + (uint32_t)ks * 2048u, SLAB, 1024);
}
constexpr uint32_t ID_KK = make_idesc(128, 128, FMT_BF16, false, false);
constexpr uint32_t ID_KM = make_idesc(128, 128, FMT_BF16, false, true);
constexpr uint32_t ID_MM = make_idesc(128, 128, FMT_BF16, true, true);
// the same products on fp16 operand tiles (both operands fp16)
constexpr uint32_t ID_KK_H = make_idesc(128, 128, FMT_F16, false, false);
constexpr uint32_t ID_KM_H = make_idesc(128, 128, FMT_F16, false, true);
constexpr uint32_t ID_MM_H = make_idesc(128, 128, FMT_F16, true, true);

// D (+)= A B^T over the 128 K of two tiles. Each operand's descriptor is formed once and offset per K
// step (the start-address field holds the byte address / 16, shared memory below 256 KB): one thread
// issues the eight MMAs about twice as fast as with a descriptor built per MMA.
__device__ __forceinline__ void mma_tile(uint32_t d, uint32_t a, bool a_mn, uint32_t b, bool b_mn, uint32_t idesc,
                                         bool acc) {
  const uint64_t da = a_mn ? mndesc(a, 0) : kdesc(a, 0), db = b_mn ? mndesc(b, 0) : kdesc(b, 0);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t oa = a_mn ? (uint32_t)ks * (2048u >> 4) : (uint32_t)((ks >> 2) * SLAB + (ks & 3) * 32) >> 4;
    const uint32_t ob = b_mn ? (uint32_t)ks * (2048u >> 4) : (uint32_t)((ks >> 2) * SLAB + (ks & 3) * 32) >> 4;
    mma_f16(d, da + oa, db + ob, idesc, (acc || ks != 0) ? 1u : 0u);
  }
}

// Wait for the MMA barrier with a CTA-uniform outcome.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, const Watch& w, int* abort_flag, int site) {
  const bool ok = wait_bounded(bar, parity, w, abort_flag, site);
  return __syncthreads_and(ok) != 0;
}

}  // namespace pt
}  // namespace tmk
