// conv1d_kernel.cuh -- depthwise conv1d rolling-buffer step.
//
// One decode step of the WGSL kernel "conv1d.wgsl" (cera 0.2.0), for a batch
// of independent sequences: for every sequence b and channel ch
//   out[b, ch] = sum_{k < d_conv} buf[b, k, ch] * w[ch, k] + x[b, ch] * w[ch, d_conv]
// (f32, taps in that order, each product-and-add one fused multiply-add),
// then buf[b, k, ch] <- buf[b, k + 1, ch] for k < d_conv - 1 and
// buf[b, d_conv - 1, ch] <- x[b, ch].  Layouts: x and out [batch, hidden],
// buf [batch, d_conv, hidden] (the page's [d_conv, hidden] per sequence),
// w [hidden, kernel_size] shared by all sequences.
//
// The step moves (2 d_conv + 2) * 4 bytes per (sequence, channel) through
// HBM and does 2 (d_conv + 1) flops on them: a pure streaming kernel.  Each
// thread owns its channels' whole buffer column, so it reads every slot
// before it writes any and no two threads touch one element.  The weights
// (hidden * kernel_size floats) are read from L1/L2 by every sequence.
#pragma once

#include <cstdint>

namespace vattn {

struct Conv1dArgs {
  const float* input;   // [batch, hidden]
  float* buffer;        // [batch, d_conv, hidden]
  const float* weight;  // [hidden, kernel_size]
  float* output;        // [batch, hidden]
  long long batch;
  int hidden;
  int kernel_size;
  int d_conv;
};

// Four consecutive channels per thread with 16-byte loads and stores;
// needs hidden % 4 == 0 and 16-byte aligned input, buffer and output.
// DC = d_conv, fixed at compile time so the slots stay in registers.
// kDense: kernel_size == d_conv + 1 and a 16-byte aligned weight, so a
// thread's 4 (d_conv + 1) taps are contiguous and come in as d_conv + 1
// 16-byte loads (4-byte loads at a lane stride of 16 (d_conv + 1) bytes hit
// the same L1 banks and cost up to a third of the bandwidth at d_conv 3).
template <int DC, bool kDense>
__global__ void __launch_bounds__(256) vattn_conv1d_step4_kernel(const Conv1dArgs a) {
  const float* __restrict__ x_base = a.input;
  float* __restrict__ buf_base = a.buffer;
  const float* __restrict__ w_base = a.weight;
  float* __restrict__ out_base = a.output;
  const int hq = a.hidden >> 2;
  const long long total = a.batch * hq;
  const int ks = a.kernel_size;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long b = idx / hq;
    const int ch = static_cast<int>(idx - b * hq) * 4;
    const float4 x = __ldcs(reinterpret_cast<const float4*>(x_base + b * a.hidden + ch));
    float4 s[DC > 0 ? DC : 1];
#pragma unroll
    for (int k = 0; k < DC; ++k)
      s[k] = __ldcs(reinterpret_cast<const float4*>(buf_base + (b * DC + k) * a.hidden + ch));
    float w[4][DC + 1];
    if constexpr (kDense) {
      // taps of channels ch .. ch + 3: 4 (DC + 1) floats from ch * (DC + 1)
      float flat[4 * (DC + 1)];
      const float4* wq = reinterpret_cast<const float4*>(w_base + static_cast<long long>(ch) * (DC + 1));
#pragma unroll
      for (int i = 0; i < DC + 1; ++i) {
        const float4 t = __ldg(wq + i);
        flat[4 * i] = t.x; flat[4 * i + 1] = t.y; flat[4 * i + 2] = t.z; flat[4 * i + 3] = t.w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int k = 0; k <= DC; ++k) w[e][k] = flat[e * (DC + 1) + k];
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int k = 0; k <= DC; ++k) w[e][k] = __ldg(w_base + static_cast<long long>(ch + e) * ks + k);
    }
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < DC; ++k) {
      acc[0] = fmaf(s[k].x, w[0][k], acc[0]);
      acc[1] = fmaf(s[k].y, w[1][k], acc[1]);
      acc[2] = fmaf(s[k].z, w[2][k], acc[2]);
      acc[3] = fmaf(s[k].w, w[3][k], acc[3]);
    }
    acc[0] = fmaf(x.x, w[0][DC], acc[0]);
    acc[1] = fmaf(x.y, w[1][DC], acc[1]);
    acc[2] = fmaf(x.z, w[2][DC], acc[2]);
    acc[3] = fmaf(x.w, w[3][DC], acc[3]);
    __stcs(reinterpret_cast<float4*>(out_base + b * a.hidden + ch),
           make_float4(acc[0], acc[1], acc[2], acc[3]));
#pragma unroll
    for (int k = 0; k + 1 < DC; ++k)
      __stcs(reinterpret_cast<float4*>(buf_base + (b * DC + k) * a.hidden + ch), s[k + 1]);
    if (DC > 0)
      __stcs(reinterpret_cast<float4*>(buf_base + (b * DC + (DC > 0 ? DC - 1 : 0)) * a.hidden + ch), x);
  }
}

// Any shape and alignment: one channel of one sequence per thread; slot k
// is read, used and written to slot k - 1 before slot k + 1 is read.
__global__ void __launch_bounds__(256) vattn_conv1d_step_kernel(const Conv1dArgs a) {
  const long long total = a.batch * a.hidden;
  const int dc = a.d_conv;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long b = idx / a.hidden;
    const int ch = static_cast<int>(idx - b * a.hidden);
    const float* w = a.weight + static_cast<long long>(ch) * a.kernel_size;
    float* col = dc > 0 ? a.buffer + b * dc * a.hidden + ch : nullptr;  // slot k at col[k * hidden]
    const float x = a.input[b * a.hidden + ch];
    float acc = 0.0f;
    for (int k = 0; k < dc; ++k) {
      const float sk = col[static_cast<long long>(k) * a.hidden];
      acc = fmaf(sk, __ldg(w + k), acc);
      if (k > 0) col[static_cast<long long>(k - 1) * a.hidden] = sk;
    }
    acc = fmaf(x, __ldg(w + dc), acc);
    a.output[b * a.hidden + ch] = acc;
    if (dc > 0) col[static_cast<long long>(dc - 1) * a.hidden] = x;
  }
}

}  // namespace vattn
