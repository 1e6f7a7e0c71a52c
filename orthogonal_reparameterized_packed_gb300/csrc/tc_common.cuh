// Pieces shared by the tcgen05 kernels: tile constants, the row epilogue,
// timeout bookkeeping and host-side tensor-map creation.
#pragma once

#include <cuda.h>

#include "internal.h"
#include "ptx.cuh"

namespace poetx {
namespace {

constexpr int BM = 128;  // MMA M: one TMEM lane per row
constexpr int BK = 64;   // one 128-byte swizzle row of bf16
constexpr int kStatusTimeout = 5;  // POETX_ERR_TIMEOUT

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  atomicCAS(status, 0, kStatusTimeout);
  *abort = 1;
}

// EPI_ROWS: one thread, one row, 32 consecutive columns.
__device__ __forceinline__ void epilogue_row32(const EpiArgs& e, int g, int s, int row, int col0,
                                               const uint32_t (&r)[32]) {
  if (row >= e.row_limit) return;
  const long long off =
      (static_cast<long long>(g) * e.row_g + static_cast<long long>(s) * e.row_s + row) * e.ld +
      static_cast<long long>(g) * e.col_g + col0;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = e.alpha * __uint_as_float(r[j]);
  if (e.X != nullptr) {
    const float4* xp = reinterpret_cast<const float4*>(e.X + off);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 t = xp[q];
      v[4 * q + 0] += e.beta * t.x;
      v[4 * q + 1] += e.beta * t.y;
      v[4 * q + 2] += e.beta * t.z;
      v[4 * q + 3] += e.beta * t.w;
    }
  }
  if (e.Y != nullptr) {
    const float4* yp = reinterpret_cast<const float4*>(e.Y + off);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 t = yp[q];
      v[4 * q + 0] += e.gamma * t.x;
      v[4 * q + 1] += e.gamma * t.y;
      v[4 * q + 2] += e.gamma * t.z;
      v[4 * q + 3] += e.gamma * t.w;
    }
  }
  if (e.delta != 0.f) {
    const int dj = row - col0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j == dj) v[j] += e.delta;
  }
  if (e.out_f32 != nullptr) {
    float4* op = reinterpret_cast<float4*>(e.out_f32 + off);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      op[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
  if (e.out_bf16 != nullptr) {
    uint4* op = reinterpret_cast<uint4*>(e.out_bf16 + off);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        __nv_bfloat162 p2 = __floats2bfloat162_rn(v[8 * q + 2 * h], v[8 * q + 2 * h + 1]);
        w[h] = *reinterpret_cast<uint32_t*>(&p2);
      }
      op[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 p2 = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&p2);
}

// ------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Resolved once per process (the static's initialiser runs once, also when
// several host threads get here at the same time).
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  return fn;
}

// 2-D map over a row-major array, box = box_cols x box_rows, 128B swizzle.
bool make_map(CUtensorMap* map, const void* ptr, long long rows, long long cols, long long pitch,
              int elem_bytes, int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * elem_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace poetx
