// stage_kernel.cuh -- the f16 staging of q, k and v, once per call.
//
// The shader "vision_attention_flash_sub_hpd_f16.wgsl" (rullama 0.1.0)
// rounds q, k and v to f16 as it copies them into workgroup storage.  Its
// workgroups re-read and re-round every key/value row once per block of 8
// queries; here each element is rounded once, into an f16 copy that the
// attention kernel then streams with TMA straight into the tensor-core
// operand layout.
//
// src: f32 [n_rows, D] (rows of all heads back to back), any alignment of 4;
// dst: f16 [n_rows, d_pad], d_pad = D rounded up to 16, columns >= D zero,
//      16-byte aligned rows (d_pad * 2 is a multiple of 32).
// Rounding: round-to-nearest-even (cvt.rn.f16x2.f32).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace vattn {

struct StageJob {
  const float* src;
  __half* dst;
};

// A walk over the 8-column chunks c = row * cpr + ch of one tensor's
// [n_rows, cpr] chunk grid: chunk c0, c0 + stride, ..., stepped by rows and
// columns so that no chunk costs a division.
struct ChunkWalk {
  long long row;
  int ch;
  long long row_step;
  int ch_step;
  __device__ __forceinline__ ChunkWalk(long long c0, long long stride, int cpr)
      : row(c0 / cpr), ch(static_cast<int>(c0 - (c0 / cpr) * cpr)), row_step(stride / cpr),
        ch_step(static_cast<int>(stride - (stride / cpr) * cpr)) {}
  __device__ __forceinline__ void next(int cpr) {
    row += row_step;
    ch += ch_step;
    if (ch >= cpr) {
      ch -= cpr;
      ++row;
    }
  }
};

// gridDim.y (2 or 3) tensors (a, b[, c]: q, k, v, or k and v alone when the
// attention kernel rounds q itself) of n_rows x D each, tensor blockIdx.y.
// Thread i of a row of blocks handles the 8-column chunks i, i + stride, ...
// of its tensor's [n_rows, d_pad / 8] chunk grid.  vec: D % 8 == 0 and
// 16-byte aligned sources -> two 16-byte loads per chunk; otherwise element
// loads.
__global__ void __launch_bounds__(256) vattn_stage_kernel(StageJob a, StageJob b, StageJob c,
                                                         long long n_rows, int D, int d_pad,
                                                         int vec) {
  const int cpr = d_pad >> 3;
  const int which = static_cast<int>(blockIdx.y);
  const StageJob job = which == 0 ? a : (which == 1 ? b : c);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (ChunkWalk w(static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x, stride, cpr);
       w.row < n_rows; w.next(cpr)) {
    const long long row = w.row;
    const int ch = w.ch;
    const float* s = job.src + row * D + ch * 8;
    float x[8];
    if (vec && ch * 8 + 8 <= D) {
      const float4 lo = __ldg(reinterpret_cast<const float4*>(s));
      const float4 hi = __ldg(reinterpret_cast<const float4*>(s) + 1);
      x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
      x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = (ch * 8 + e < D) ? __ldg(s + e) : 0.0f;
    }
    uint4 h;
    h.x = ptx::pack_half2(x[0], x[1]);
    h.y = ptx::pack_half2(x[2], x[3]);
    h.z = ptx::pack_half2(x[4], x[5]);
    h.w = ptx::pack_half2(x[6], x[7]);
    *reinterpret_cast<uint4*>(job.dst + row * d_pad + ch * 8) = h;
  }
  ptx::grid_dep_launch();  // the attention kernel may launch once every block got here
}

}  // namespace vattn

namespace vattn {

// Two-term f16 split of q, k and v for the accurate mode:
//   hi = f16(x), lo = f16(x - f32(hi))   (round to nearest even both times)
// so x = hi + lo to about 2^-22 relative (f16 subnormals bound lo's error
// at 2^-25 absolute).  Same layout, grid and chunk walk as
// vattn_stage_kernel; `dst` of each job receives hi, `dst_lo` lo.
struct SplitJob {
  const float* src;
  __half* dst;
  __half* dst_lo;
};

__global__ void __launch_bounds__(256) vattn_stage_split_kernel(SplitJob a, SplitJob b, SplitJob c,
                                                               long long n_rows, int D, int d_pad,
                                                               int vec) {
  const int cpr = d_pad >> 3;
  const int which = static_cast<int>(blockIdx.y);  // gridDim.y = 3: q, k, v
  const SplitJob job = which == 0 ? a : (which == 1 ? b : c);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (ChunkWalk w(static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x, stride, cpr);
       w.row < n_rows; w.next(cpr)) {
    const long long row = w.row;
    const int ch = w.ch;
    const float* s = job.src + row * D + ch * 8;
    float x[8];
    if (vec && ch * 8 + 8 <= D) {
      const float4 lo = __ldg(reinterpret_cast<const float4*>(s));
      const float4 hi = __ldg(reinterpret_cast<const float4*>(s) + 1);
      x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
      x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = (ch * 8 + e < D) ? __ldg(s + e) : 0.0f;
    }
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h[e] = ptx::pack_half2(x[2 * e], x[2 * e + 1]);
      const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
      l[e] = ptx::pack_half2(x[2 * e] - back.x, x[2 * e + 1] - back.y);
    }
    *reinterpret_cast<uint4*>(job.dst + row * d_pad + ch * 8) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(job.dst_lo + row * d_pad + ch * 8) = make_uint4(l[0], l[1], l[2], l[3]);
  }
  ptx::grid_dep_launch();  // the attention kernel may launch once every block got here
}

}  // namespace vattn
