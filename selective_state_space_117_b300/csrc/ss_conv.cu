// Causal depthwise convolution of width 4 with an optional SiLU (the short
// convolution in front of the selective SSM in a Mamba block).
//
//   out[b,d,t] = silu(bias[d] + sum_{k=0..3} w[d,k] * x[b,d,t-3+k]),  x = 0 before t = 0
//
// A warp walks one row (b, d) over a segment of kSegWindows windows of 256
// steps: lane l loads steps 8l..8l+7 of the window as one 16-byte (bf16) or
// two 16-byte (fp32) vectors, so the warp reads and writes contiguous runs.
// The three steps before a lane's chunk come from its left neighbour by
// shuffle, and lane 0 takes them from lane 31 of the previous window (or from
// memory at the start of a segment).  Memory-bound: 2 x (element size) bytes
// of traffic per element.
#include <cuda_bf16.h>

#include "ss_device.cuh"
#include "ss_launch.h"

namespace ssk {

constexpr int kConvThreads = 256;
constexpr int kSegWindows = 32;   // windows of 256 steps per warp

template <bool BF>
__device__ __forceinline__ void store8(void* out, int64_t i, const float (&v)[8]) {
  if (BF) {
    uint4 w;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]), p1 = __floats2bfloat162_rn(v[2], v[3]);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(v[4], v[5]), p3 = __floats2bfloat162_rn(v[6], v[7]);
    w.x = *reinterpret_cast<uint32_t*>(&p0);
    w.y = *reinterpret_cast<uint32_t*>(&p1);
    w.z = *reinterpret_cast<uint32_t*>(&p2);
    w.w = *reinterpret_cast<uint32_t*>(&p3);
    *reinterpret_cast<uint4*>(static_cast<unsigned short*>(out) + i) = w;
  } else {
    float4* q = reinterpret_cast<float4*>(static_cast<float*>(out) + i);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

template <bool BF>
__device__ __forceinline__ void store1(void* out, int64_t i, float v) {
  if (BF) static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else static_cast<float*>(out)[i] = v;
}

template <bool BF, bool SILU>
__global__ void __launch_bounds__(kConvThreads) conv1d_kernel(const ConvArgs a) {
  using L = In<BF>;
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * kConvThreads + threadIdx.x) >> 5;   // global warp
  const int64_t row = gw / a.nseg, seg = gw % a.nseg;
  if (row >= a.rows) return;                       // whole warps leave together
  const int64_t d = row % a.dim;
  const int64_t base = row * a.seqlen;
  // Debug build: the row and the channel's taps.
  if (!span_ok(a.err, base, a.seqlen, a.rows * a.seqlen) || !span_ok(a.err, d * 4, 4, a.dim * 4)) return;
  const float4 w = *reinterpret_cast<const float4*>(a.w + d * 4);
  const float bias = a.bias ? a.bias[d] : 0.f;
  const int64_t t_seg = seg * (int64_t)kSegWindows * 256;
  const int64_t t_end = min(a.seqlen, t_seg + (int64_t)kSegWindows * 256);

  // The three steps before the segment.
  float h1 = 0.f, h2 = 0.f, h3 = 0.f;               // x[t-3], x[t-2], x[t-1] for lane 0
  if (t_seg > 0) {
    h1 = L::one(a.x, base + t_seg - 3);
    h2 = L::one(a.x, base + t_seg - 2);
    h3 = L::one(a.x, base + t_seg - 1);
  }
  for (int64_t w0 = t_seg; w0 < t_end; w0 += 256) {
    const int64_t t = w0 + 8 * lane;
    float v[8];
    const bool full = a.vec && t + 8 <= t_end;
    if (full) {
      const typename L::Raw8 r = L::load8(a.x, base + t);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const f2 q = L::pair(r, p);
        v[2 * p] = lo(q);
        v[2 * p + 1] = hi(q);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = (t + j < t_end) ? L::one(a.x, base + t + j) : 0.f;
    }
    // x[t-3..t-1]: the left neighbour's last three steps; lane 0 keeps the carry.
    float p1 = __shfl_up_sync(0xffffffffu, v[5], 1);
    float p2 = __shfl_up_sync(0xffffffffu, v[6], 1);
    float p3 = __shfl_up_sync(0xffffffffu, v[7], 1);
    if (lane == 0) {
      p1 = h1;
      p2 = h2;
      p3 = h3;
    }
    h1 = __shfl_sync(0xffffffffu, v[5], 31);
    h2 = __shfl_sync(0xffffffffu, v[6], 31);
    h3 = __shfl_sync(0xffffffffu, v[7], 31);
    const float xs[11] = {p1, p2, p3, v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]};
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float s = fmaf(w.x, xs[j], bias);
      s = fmaf(w.y, xs[j + 1], s);
      s = fmaf(w.z, xs[j + 2], s);
      s = fmaf(w.w, xs[j + 3], s);
      o[j] = SILU ? silu(s) : s;
    }
    if (full) {
      store8<BF>(a.out, base + t, o);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (t + j < t_end) store1<BF>(a.out, base + t + j, o[j]);
    }
  }
}

int launch_conv1d(const ConvArgs& a, bool bf16, bool silu_on, cudaStream_t s) {
  const int64_t warps = a.rows * a.nseg;
  const int64_t blocks = (warps * 32 + kConvThreads - 1) / kConvThreads;
  if (blocks > 2147483647) return -1;
  if (bf16) {
    if (silu_on) conv1d_kernel<true, true><<<(unsigned)blocks, kConvThreads, 0, s>>>(a);
    else conv1d_kernel<true, false><<<(unsigned)blocks, kConvThreads, 0, s>>>(a);
  } else {
    if (silu_on) conv1d_kernel<false, true><<<(unsigned)blocks, kConvThreads, 0, s>>>(a);
    else conv1d_kernel<false, false><<<(unsigned)blocks, kConvThreads, 0, s>>>(a);
  }
  return 0;
}

int64_t conv1d_segments(int64_t seqlen) { return (seqlen + kSegWindows * 256 - 1) / (kSegWindows * 256); }

}  // namespace ssk
