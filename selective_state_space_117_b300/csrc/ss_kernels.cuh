// Selective scan kernels (sm_103a).
//
// Work decomposition: one thread owns one (batch row b, channel d, chunk k)
// and keeps that channel's N states in registers for the whole chunk, so the
// (batch, L, dim, N) expanded state never leaves the SM ("Kernel fusion",
// "Mamba: Linear-Time Sequence Modeling with Selective State Spaces").  A
// block is 128 consecutive channels of one (b, k); all of them read the same
// B_t and C_t, which the block stages through shared memory one time tile at
// a time and every thread then reads as broadcast float4 loads.  u, delta and
// z are read along each thread's own row with 16-byte vector loads (8 steps
// per load for bf16, 2 loads for fp32); y is written the same way.
//
// Modes:
//   kFull   start from h = 0, write y and (optionally) the final state
//   kLocal  start from h = 0, write only the chunk's end state and sum(dt)
//   kFixup  start from the carried-in state in the workspace, write y
#pragma once

#include "ss_device.cuh"
#include "ss_types.h"

namespace ssk {

template <int NT, bool BF, bool HAS_Z, int MODE>
__global__ void __launch_bounds__(kThreads) scan_kernel(const ScanArgs a) {
  using L = In<BF>;
  __shared__ __align__(16) float sB[kTile][NT + 4];
  __shared__ __align__(16) float sC[MODE == kLocal ? 1 : kTile][NT + 4];

  const int tid = threadIdx.x;
  const int ct = blockIdx.x % a.ctiles;
  const int64_t k = blockIdx.x / a.ctiles;
  const int64_t b = blockIdx.y;
  const int64_t d = (int64_t)ct * kThreads + tid;
  const bool active = d < a.dim;
  const int N = (int)a.dstate;
  const int64_t Lq = a.seqlen;
  const int64_t t_begin = k * a.chunk_len;
  const int64_t t_end = min(Lq, t_begin + a.chunk_len);

  // Padding states n >= N read B = C = 0 forever, so they stay 0 and add nothing.
  for (int i = tid; i < kTile * (NT + 4); i += kThreads) {
    (&sB[0][0])[i] = 0.f;
    if (MODE != kLocal) (&sC[0][0])[i] = 0.f;
  }

  float A2[NT], h[NT];
  const int64_t bd = b * a.dim + (active ? d : 0);
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    A2[n] = (active && n < N) ? a.A[(active ? d : 0) * N + n] * kLog2e : 0.f;
    h[n] = 0.f;
    if (MODE == kFixup && active && n < N) h[n] = a.ws_H[(bd * a.nchunks + k) * N + n];
  }
  const float bias = (a.delta_bias && active) ? a.delta_bias[d] : 0.f;
  const float Dd = (a.D && active) ? a.D[d] : 0.f;
  const int64_t row = bd * Lq;                   // (b, d, 0)
  const int64_t bc_row = b * (int64_t)N * Lq;    // (b, 0, 0)
  float S = 0.f;

  for (int64_t tt0 = t_begin; tt0 < t_end; tt0 += kTile) {
    __syncthreads();
    const int tn = (int)min((int64_t)kTile, t_end - tt0);
    for (int i = tid; i < N * kTile; i += kThreads) {
      const int n = i / kTile, j = i % kTile;
      if (j < tn) {
        const int64_t off = bc_row + (int64_t)n * Lq + tt0 + j;
        sB[j][n] = L::one(a.B, off);
        if (MODE != kLocal) sC[j][n] = L::one(a.C, off);
      }
    }
    __syncthreads();
    if (!active) continue;

    float Ssub = 0.f;
    for (int g = 0; g < tn; g += kGroup) {
      const int64_t t = tt0 + g;
      const int nv = min(kGroup, tn - g);
      float uu[kGroup], dr[kGroup], zz[kGroup];
      if (nv == kGroup && a.vec) {
        L::eight(a.u, row + t, uu);
        L::eight(a.delta, row + t, dr);
        if (HAS_Z && MODE != kLocal) L::eight(a.z, row + t, zz);
      } else {
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          const bool ok = j < nv;
          uu[j] = ok ? L::one(a.u, row + t + j) : 0.f;
          dr[j] = ok ? L::one(a.delta, row + t + j) : 0.f;
          zz[j] = (HAS_Z && MODE != kLocal && ok) ? L::one(a.z, row + t + j) : 0.f;
        }
      }
      float yo[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        yo[j] = 0.f;
        if (j < nv) {
          const float x = dr[j] + bias;
          const float dt = a.softplus ? softplus(x) : x;
          const float du = dt * uu[j];
          const int js = g + j;
          if (MODE == kLocal) {
            Ssub += dt;
#pragma unroll
            for (int n4 = 0; n4 < NT; n4 += 4) {
              const float4 bv = *reinterpret_cast<const float4*>(&sB[js][n4]);
              h[n4 + 0] = fmaf(ex2(dt * A2[n4 + 0]), h[n4 + 0], du * bv.x);
              h[n4 + 1] = fmaf(ex2(dt * A2[n4 + 1]), h[n4 + 1], du * bv.y);
              h[n4 + 2] = fmaf(ex2(dt * A2[n4 + 2]), h[n4 + 2], du * bv.z);
              h[n4 + 3] = fmaf(ex2(dt * A2[n4 + 3]), h[n4 + 3], du * bv.w);
            }
          } else {
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int n4 = 0; n4 < NT; n4 += 4) {
              const float4 bv = *reinterpret_cast<const float4*>(&sB[js][n4]);
              const float4 cv = *reinterpret_cast<const float4*>(&sC[js][n4]);
              h[n4 + 0] = fmaf(ex2(dt * A2[n4 + 0]), h[n4 + 0], du * bv.x);
              h[n4 + 1] = fmaf(ex2(dt * A2[n4 + 1]), h[n4 + 1], du * bv.y);
              h[n4 + 2] = fmaf(ex2(dt * A2[n4 + 2]), h[n4 + 2], du * bv.z);
              h[n4 + 3] = fmaf(ex2(dt * A2[n4 + 3]), h[n4 + 3], du * bv.w);
              acc0 = fmaf(cv.x, h[n4 + 0], acc0);
              acc1 = fmaf(cv.y, h[n4 + 1], acc1);
              acc0 = fmaf(cv.z, h[n4 + 2], acc0);
              acc1 = fmaf(cv.w, h[n4 + 3], acc1);
            }
            float yv = fmaf(Dd, uu[j], acc0 + acc1);
            if (HAS_Z) yv *= silu(zz[j]);
            yo[j] = yv;
          }
        }
      }
      if (MODE != kLocal) {
        if (nv == kGroup && a.vec) {
          float4* q = reinterpret_cast<float4*>(a.y + row + t);
          q[0] = make_float4(yo[0], yo[1], yo[2], yo[3]);
          q[1] = make_float4(yo[4], yo[5], yo[6], yo[7]);
        } else {
#pragma unroll
          for (int j = 0; j < kGroup; ++j)
            if (j < nv) a.y[row + t + j] = yo[j];
        }
      }
    }
    S += Ssub;
  }

  if (!active) return;
  if (MODE == kFull && a.last_state) {
#pragma unroll
    for (int n = 0; n < NT; ++n)
      if (n < N) a.last_state[bd * N + n] = h[n];
  }
  if (MODE == kLocal) {
    a.ws_S[bd * a.nchunks + k] = S;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      if (n < N) a.ws_H[(bd * a.nchunks + k) * N + n] = h[n];
  }
}

}  // namespace ssk
