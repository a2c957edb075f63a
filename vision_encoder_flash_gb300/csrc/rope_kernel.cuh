// rope_kernel.cuh -- NeoX rotary embedding (RoPE) on head-major tensors.
//
// The rotation of the WGSL kernel "rope_neox_backward.wgsl" (rullama 0.2.0):
// with half = rope_dims / 2, every pair (x[i], x[i + half]), i < half, of a
// head is turned by theta_i = pos * base^(-2 i / rope_dims) (divided by
// factors[i] when a factor table is given):
//   forward  x[i] <- a cos - b sin,  x[i + half] <- a sin + b cos
//   inverse  x[i] <- a cos + b sin,  x[i + half] <- -a sin + b cos
// and dims >= 2 * half are left alone.  The page rotates the heads of one
// token; here the tensors are [batch*heads, n_patches, head_dim] and patch n
// sits at position pos0 + n.
//
// theta, cos and sin depend on (patch, pair) only, so one small kernel
// fills a table [n_patches][half] of (cos, sin) once per call, computed in
// f32 in the page's order (f32(pos) * pow(base, -2 i / rope_dims), then
// / factors[i]); the passes over the tensors read it (it stays in L2).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "stage_kernel.cuh"

namespace vattn {

__global__ void __launch_bounds__(256) vattn_rope_table_kernel(float2* tab, int n_patches,
                                                              int half, int rope_dims,
                                                              long long pos0, float base,
                                                              const float* factors) {
  const long long total = static_cast<long long>(n_patches) * half;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(idx / half);
    const int i = static_cast<int>(idx - static_cast<long long>(n) * half);
    const float exp_v = -2.0f * static_cast<float>(i) / static_cast<float>(rope_dims);
    float theta = static_cast<float>(pos0 + n) * powf(base, exp_v);
    if (factors != nullptr) theta = theta / factors[i];
    tab[idx] = make_float2(cosf(theta), sinf(theta));
  }
}

// In place on x [n_rows, D], row r at patch r % n_patches, four pairs per
// thread with 16-byte accesses; needs half % 4 == 0, D % 4 == 0 and a 16-byte
// aligned x.
__global__ void __launch_bounds__(256) vattn_rope_apply4_kernel(float* x, long long n_rows,
                                                               int n_patches, int D, int half,
                                                               const float2* tab, int inverse) {
  const int quads = half >> 2;
  const long long total = n_rows * quads;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = idx / quads;
    const int i = static_cast<int>(idx - row * quads) * 4;
    const float4* t = reinterpret_cast<const float4*>(tab + (row % n_patches) * half + i);
    const float4 cs01 = __ldg(t), cs23 = __ldg(t + 1);
    const float c[4] = {cs01.x, cs01.z, cs23.x, cs23.z};
    const float sn[4] = {cs01.y, cs01.w, cs23.y, cs23.w};
    float4* pa = reinterpret_cast<float4*>(x + row * D + i);
    float4* pb = reinterpret_cast<float4*>(x + row * D + i + half);
    const float4 a4 = *pa, b4 = *pb;
    const float a[4] = {a4.x, a4.y, a4.z, a4.w}, b[4] = {b4.x, b4.y, b4.z, b4.w};
    float ra[4], rb[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!inverse) {
        ra[e] = a[e] * c[e] - b[e] * sn[e];
        rb[e] = a[e] * sn[e] + b[e] * c[e];
      } else {
        ra[e] = a[e] * c[e] + b[e] * sn[e];
        rb[e] = -a[e] * sn[e] + b[e] * c[e];
      }
    }
    *pa = make_float4(ra[0], ra[1], ra[2], ra[3]);
    *pb = make_float4(rb[0], rb[1], rb[2], rb[3]);
  }
}

// In place on x [n_rows, D], row r at patch r % n_patches; one thread per
// (row, pair) (any shape).
__global__ void __launch_bounds__(256) vattn_rope_apply_kernel(float* x, long long n_rows,
                                                              int n_patches, int D, int half,
                                                              const float2* tab, int inverse) {
  const long long total = n_rows * half;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = idx / half;
    const int i = static_cast<int>(idx - row * half);
    const int n = static_cast<int>(row % n_patches);
    const float2 cs = tab[static_cast<long long>(n) * half + i];
    float* r = x + row * D;
    const float a = r[i];
    const float b = r[i + half];
    if (!inverse) {
      r[i] = a * cs.x - b * cs.y;
      r[i + half] = a * cs.y + b * cs.x;
    } else {
      r[i] = a * cs.x + b * cs.y;
      r[i + half] = -a * cs.y + b * cs.x;
    }
  }
}

// The f16 staging of vattn_stage_kernel with q and k (jobs a and b) turned
// forward by the table's angles before rounding; v (job c) is only
// converted.  Same chunk decomposition: thread = 8 output columns of one row.
__global__ void __launch_bounds__(256) vattn_stage_rope_kernel(StageJob a, StageJob b, StageJob c,
                                                              long long n_rows, int n_patches,
                                                              int D, int d_pad, int half,
                                                              const float2* tab, int vec) {
  const int cpr = d_pad >> 3;
  const long long chunks_per_tensor = n_rows * cpr;
  const long long total = 3 * chunks_per_tensor;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // vectorised pairs of chunks: half a multiple of 8 (so every rotated chunk
  // is whole and lies inside the row) and 16-byte loads
  const bool pair_chunks = vec && (half & 7) == 0;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += stride) {
    const int which = static_cast<int>(idx / chunks_per_tensor);
    const long long r = idx - which * chunks_per_tensor;
    const long long row = r / cpr;
    const int ch = static_cast<int>(r - row * cpr);
    // in the paired mode a partner chunk (half / 8 <= ch < half / 4) is
    // done by the thread of chunk ch - half / 8
    if (which < 2 && pair_chunks && ch * 8 >= half && ch * 8 < 2 * half) continue;
    const StageJob job = which == 0 ? a : (which == 1 ? b : c);
    const float* s = job.src + row * D;
    float x[8];
    if (vec && ch * 8 + 8 <= D) {
      const float4 lo = __ldg(reinterpret_cast<const float4*>(s + ch * 8));
      const float4 hi = __ldg(reinterpret_cast<const float4*>(s + ch * 8) + 1);
      x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
      x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = (ch * 8 + e < D) ? __ldg(s + ch * 8 + e) : 0.0f;
    }
    if (which < 2 && pair_chunks && ch * 8 < half) {
      // chunk ch together with its partner ch + half / 8
      const int chb = ch + (half >> 3);
      const float4 lo = __ldg(reinterpret_cast<const float4*>(s + chb * 8));
      const float4 hi = __ldg(reinterpret_cast<const float4*>(s + chb * 8) + 1);
      const float y[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      const float4* t = reinterpret_cast<const float4*>(
          tab + static_cast<long long>(row % n_patches) * half + ch * 8);
      float ra[8], rb[8];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 cs = __ldg(t + q4);  // (cos, sin) of pairs 2 q4 and 2 q4 + 1
        ra[2 * q4] = x[2 * q4] * cs.x - y[2 * q4] * cs.y;
        rb[2 * q4] = x[2 * q4] * cs.y + y[2 * q4] * cs.x;
        ra[2 * q4 + 1] = x[2 * q4 + 1] * cs.z - y[2 * q4 + 1] * cs.w;
        rb[2 * q4 + 1] = x[2 * q4 + 1] * cs.w + y[2 * q4 + 1] * cs.z;
      }
      uint4 ha, hb;
      ha.x = ptx::pack_half2(ra[0], ra[1]); ha.y = ptx::pack_half2(ra[2], ra[3]);
      ha.z = ptx::pack_half2(ra[4], ra[5]); ha.w = ptx::pack_half2(ra[6], ra[7]);
      hb.x = ptx::pack_half2(rb[0], rb[1]); hb.y = ptx::pack_half2(rb[2], rb[3]);
      hb.z = ptx::pack_half2(rb[4], rb[5]); hb.w = ptx::pack_half2(rb[6], rb[7]);
      *reinterpret_cast<uint4*>(job.dst + row * d_pad + ch * 8) = ha;
      *reinterpret_cast<uint4*>(job.dst + row * d_pad + chb * 8) = hb;
      continue;
    }
    if (which < 2 && ch * 8 < 2 * half) {
      const float2* t = tab + static_cast<long long>(row % n_patches) * half;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int d = ch * 8 + e;
        if (d < half) {  // x[i] <- a cos - b sin, b = x[i + half]
          const float2 cs = __ldg(t + d);
          x[e] = x[e] * cs.x - __ldg(s + d + half) * cs.y;
        } else if (d < 2 * half) {  // x[i + half] <- a sin + b cos, a = x[i]
          const float2 cs = __ldg(t + d - half);
          x[e] = __ldg(s + d - half) * cs.y + x[e] * cs.x;
        }
      }
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
