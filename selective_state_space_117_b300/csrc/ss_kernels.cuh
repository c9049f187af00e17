// Selective scan kernels (sm_103a).
//
// Work decomposition: one thread owns one (batch row b, channel d, chunk k)
// and keeps that channel's N states in registers for the whole chunk, so the
// (batch, L, dim, N) expanded state never leaves the SM ("Kernel fusion",
// "Mamba: Linear-Time Sequence Modeling with Selective State Spaces").  A
// block is 128 consecutive channels of one (b, k).  All of them read the same
// B_t and C_t, which the block stages through shared memory (converted to
// fp32, double-buffered: the next tile is loaded into registers while the
// current one is consumed) and every thread reads as broadcast 16-byte loads.
// u, delta and z are read along each thread's own row with 16-byte vector
// loads, one group of 8 steps ahead of use; y is written the same way.
//
// Arithmetic runs on state pairs with the packed f32x2 instructions: per
// pair and step one mul (dt*A), two MUFU.EX2, one mul (du*B), one fma (the
// state) and one fma (the readout C*h).
//
// Modes of scan_kernel:
//   kFull   start from h = 0, write y and (optionally) the final state
//   kFixup  start from the carried-in state in the workspace, write y
// local_kernel is the first phase of the chunked scan (see its comment).
#pragma once

#include "ss_device.cuh"
#include "ss_types.h"

namespace ssk {

// Time steps per shared-memory tile: NT * tile = 1024 keeps the staging work
// at 8 values per thread and array for every state count.
template <int NT>
struct TileOf {
  static constexpr int kSteps = 1024 / NT;
  static constexpr int kRow = NT + 4;  // fp32 row stride: a 16-byte multiple
  static constexpr int kPerThread = NT * kSteps / kThreads;
};

// Cooperative load of one tile of B (and C) rows [tt0, tt0 + tn) into registers,
// and its store (transposed to [t][n], fp32) into shared memory.
template <int NT, bool BF, bool WITH_C>
struct Stager {
  using L = In<BF>;
  using T = TileOf<NT>;
  float b[T::kPerThread], c[WITH_C ? T::kPerThread : 1];

  __device__ __forceinline__ void load(const ScanArgs& a, int64_t bc_row, int64_t tt0, int tn, int N, int tid) {
#pragma unroll
    for (int k = 0; k < T::kPerThread; ++k) {
      const int e = tid + k * kThreads;
      const int n = e / T::kSteps, j = e % T::kSteps;
      const bool ok = n < N && j < tn;
      const int64_t off = bc_row + (int64_t)n * a.seqlen + tt0 + j;
      b[k] = ok ? L::one(a.B, off) : 0.f;
      if (WITH_C) c[k] = ok ? L::one(a.C, off) : 0.f;
    }
  }
  __device__ __forceinline__ void store(float* sB, float* sC, int tid) const {
#pragma unroll
    for (int k = 0; k < T::kPerThread; ++k) {
      const int e = tid + k * kThreads;
      const int n = e / T::kSteps, j = e % T::kSteps;
      sB[j * T::kRow + n] = b[k];
      if (WITH_C) sC[j * T::kRow + n] = c[k];
    }
  }
};

template <int NT, bool BF, bool HAS_Z, int MODE>
__global__ void __launch_bounds__(kThreads) scan_kernel(const ScanArgs a) {
  using L = In<BF>;
  using T = TileOf<NT>;
  constexpr int NP = NT / 2;
  __shared__ __align__(16) float sB[2][T::kSteps * T::kRow];
  __shared__ __align__(16) float sC[2][T::kSteps * T::kRow];

  const int tid = threadIdx.x;
  const int ct = blockIdx.x % a.ctiles;
  const int64_t k = blockIdx.x / a.ctiles;
  const int64_t b = blockIdx.y;
  const int64_t d = (int64_t)ct * kThreads + tid;
  const bool active = d < a.dim;
  const int N = (int)a.dstate;
  const int64_t t_begin = k * a.chunk_len;
  const int64_t t_end = min(a.seqlen, t_begin + a.chunk_len);
  const int64_t bd = b * a.dim + (active ? d : 0);
  const int64_t row = bd * a.seqlen;                 // (b, d, 0)
  const int64_t bc_row = b * (int64_t)N * a.seqlen;  // (b, 0, 0)

  // Padding states n >= N keep B = C = 0 (their staged values are zero), A = 0 and h = 0.
  f2 A2[NP], h[NP];
  const float* Arow = a.A + (active ? d : 0) * N;
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int n0 = 2 * q, n1 = 2 * q + 1;
    A2[q] = pk((active && n0 < N) ? Arow[n0] * kLog2e : 0.f, (active && n1 < N) ? Arow[n1] * kLog2e : 0.f);
    float h0 = 0.f, h1 = 0.f;
    if (MODE == kFixup && active) {
      const float* H = a.ws_H + (bd * a.nchunks + k) * N;
      if (n0 < N) h0 = H[n0];
      if (n1 < N) h1 = H[n1];
    }
    h[q] = pk(h0, h1);
  }
  const float bias = (a.delta_bias && active) ? a.delta_bias[d] : 0.f;
  const float Dd = (a.D && active) ? a.D[d] : 0.f;
  const f2 bias2 = pk(bias, bias), D2 = pk(Dd, Dd);

  // Prefetch of the first group of 8 steps (vector path only).
  typename L::Raw8 ru{}, rd{}, rz{};
  bool have = active && a.vec && t_begin + kGroup <= t_end;
  if (have) {
    ru = L::load8(a.u, row + t_begin);
    rd = L::load8(a.delta, row + t_begin);
    if (HAS_Z) rz = L::load8(a.z, row + t_begin);
  }

  Stager<NT, BF, true> st;
  st.load(a, bc_row, t_begin, (int)min((int64_t)T::kSteps, t_end - t_begin), N, tid);
  st.store(sB[0], sC[0], tid);
  __syncthreads();

  int buf = 0;
  for (int64_t tt0 = t_begin; tt0 < t_end; tt0 += T::kSteps) {
    const int tn = (int)min((int64_t)T::kSteps, t_end - tt0);
    const int64_t nx0 = tt0 + T::kSteps;
    const bool more = nx0 < t_end;
    if (more) st.load(a, bc_row, nx0, (int)min((int64_t)T::kSteps, t_end - nx0), N, tid);

    if (active) {
      const float* cB = sB[buf];
      const float* cC = sC[buf];
      for (int g = 0; g < tn; g += kGroup) {
        const int64_t t = tt0 + g;
        const int nv = min(kGroup, tn - g);
        // ---- this group's inputs as pairs
        f2 u2[4], x2[4], z2[4];
        if (have) {
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            u2[p] = L::pair(ru, p);
            x2[p] = L::pair(rd, p);
            z2[p] = HAS_Z ? L::pair(rz, p) : pk(0.f, 0.f);
          }
        } else {
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            float v[3][2];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              const int j = 2 * p + s;
              const bool ok = j < nv;
              v[0][s] = ok ? L::one(a.u, row + t + j) : 0.f;
              v[1][s] = ok ? L::one(a.delta, row + t + j) : 0.f;
              v[2][s] = (HAS_Z && ok) ? L::one(a.z, row + t + j) : 0.f;
            }
            u2[p] = pk(v[0][0], v[0][1]);
            x2[p] = pk(v[1][0], v[1][1]);
            z2[p] = pk(v[2][0], v[2][1]);
          }
        }
        // ---- prefetch the next group
        const int64_t tq = t + kGroup;
        have = a.vec && tq + kGroup <= t_end;
        if (have) {
          ru = L::load8(a.u, row + tq);
          rd = L::load8(a.delta, row + tq);
          if (HAS_Z) rz = L::load8(a.z, row + tq);
        }
        // ---- per-step scalars for the group
        f2 dt2[4], du2[4], y2[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const f2 x = add2(x2[p], bias2);
          dt2[p] = a.softplus ? softplus2(x) : x;
          du2[p] = mul2(dt2[p], u2[p]);
          y2[p] = mul2(D2, u2[p]);
        }
        // ---- the recurrence, one step at a time
        float yo[kGroup];
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          yo[j] = 0.f;
          if (j < nv) {
            const float dt = (j & 1) ? hi(dt2[j >> 1]) : lo(dt2[j >> 1]);
            const float du = (j & 1) ? hi(du2[j >> 1]) : lo(du2[j >> 1]);
            const f2 dtp = pk(dt, dt), dup = pk(du, du);
            f2 acc = pk((j & 1) ? hi(y2[j >> 1]) : lo(y2[j >> 1]), 0.f);
            const float* rb = cB + (g + j) * T::kRow;
            const float* rc = cC + (g + j) * T::kRow;
#pragma unroll
            for (int q = 0; q < NP; q += 2) {
              const float4 bv = *reinterpret_cast<const float4*>(rb + 2 * q);
              const float4 cv = *reinterpret_cast<const float4*>(rc + 2 * q);
              const f2 e0 = ex2x2(mul2(dtp, A2[q]));
              h[q] = fma2(e0, h[q], mul2(dup, pk(bv.x, bv.y)));
              acc = fma2(pk(cv.x, cv.y), h[q], acc);
              const f2 e1 = ex2x2(mul2(dtp, A2[q + 1]));
              h[q + 1] = fma2(e1, h[q + 1], mul2(dup, pk(bv.z, bv.w)));
              acc = fma2(pk(cv.z, cv.w), h[q + 1], acc);
            }
            yo[j] = lo(acc) + hi(acc);
          }
        }
        if (HAS_Z) {
#pragma unroll
          for (int j = 0; j < kGroup; ++j) {
            const float z = (j & 1) ? hi(z2[j >> 1]) : lo(z2[j >> 1]);
            yo[j] *= silu(z);
          }
        }
        if (nv == kGroup && a.vec) {
          float4* qy = reinterpret_cast<float4*>(a.y + row + t);
          qy[0] = make_float4(yo[0], yo[1], yo[2], yo[3]);
          qy[1] = make_float4(yo[4], yo[5], yo[6], yo[7]);
        } else {
#pragma unroll
          for (int j = 0; j < kGroup; ++j)
            if (j < nv) a.y[row + t + j] = yo[j];
        }
      }
    }
    if (more) {
      st.store(sB[buf ^ 1], sC[buf ^ 1], tid);
      __syncthreads();
      buf ^= 1;
    }
  }

  if (MODE == kFull && active && a.last_state) {
    float* out = a.last_state + bd * N;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      if (2 * q < N) out[2 * q] = lo(h[q]);
      if (2 * q + 1 < N) out[2 * q + 1] = hi(h[q]);
    }
  }
}

// First phase of the chunked scan: for every chunk, its zero-start end state
//   Hend[n] = sum_s exp(A[n] * R_s) * dt_s * B_s[n] * u_s,   R_s = sum_{r > s in chunk} dt_r
// and the chunk's sum of dt, computed backward from the chunk's end.  With
// dt >= 0 (softplus on) R only grows, so once A[n] * R * log2(e) < -127 every
// remaining weight exp2(.) of state n is below 2^-127 and flushes to zero in
// fp32: such state pairs are skipped (per warp, per tile), and the loop stops
// once no pair in the block is left.  The sum written is then partial, but
// every exp(A[n] * sum) that the carry pass forms from it underflows to zero
// exactly as the full sum's would.
template <int NT, bool BF>
__global__ void __launch_bounds__(kThreads) local_kernel(const ScanArgs a) {
  using L = In<BF>;
  using T = TileOf<NT>;
  constexpr int NP = NT / 2;
  constexpr float kDead = -127.f;
  __shared__ __align__(16) float sB[T::kSteps * T::kRow];

  const int tid = threadIdx.x;
  const int ct = blockIdx.x % a.ctiles;
  const int64_t k = blockIdx.x / a.ctiles;
  const int64_t b = blockIdx.y;
  const int64_t d = (int64_t)ct * kThreads + tid;
  const bool active = d < a.dim;
  const int N = (int)a.dstate;
  const int64_t t_begin = k * a.chunk_len;
  const int64_t t_end = min(a.seqlen, t_begin + a.chunk_len);
  const int64_t bd = b * a.dim + (active ? d : 0);
  const int64_t row = bd * a.seqlen;
  const int64_t bc_row = b * (int64_t)N * a.seqlen;

  f2 A2[NP], acc[NP];
  float amax[NP];
  const float* Arow = a.A + (active ? d : 0) * N;
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int n0 = 2 * q, n1 = 2 * q + 1;
    const float a0 = (active && n0 < N) ? Arow[n0] * kLog2e : 0.f;
    const float a1 = (active && n1 < N) ? Arow[n1] * kLog2e : 0.f;
    A2[q] = pk(a0, a1);
    // padding states never keep a pair alive
    amax[q] = fmaxf(n0 < N ? a0 : -1e30f, n1 < N ? a1 : -1e30f);
    acc[q] = pk(0.f, 0.f);
  }
  const float bias = (a.delta_bias && active) ? a.delta_bias[d] : 0.f;
  const f2 bias2 = pk(bias, bias);
  const bool may_stop = a.softplus != 0;
  float R = 0.f;

  const int64_t ntiles = (t_end - t_begin + T::kSteps - 1) / T::kSteps;
  for (int64_t it = ntiles - 1; it >= 0; --it) {
    const int64_t tt0 = t_begin + it * T::kSteps;
    const int tn = (int)min((int64_t)T::kSteps, t_end - tt0);
    // which pairs can still receive a non-zero weight in this tile (R only grows backward)
    unsigned live = 0;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const bool mine = active && !(may_stop && amax[q] * R < kDead);
      if (__any_sync(0xffffffffu, mine)) live |= 1u << q;
    }
    if (!__syncthreads_or(live != 0)) break;
    Stager<NT, BF, false> st;
    st.load(a, bc_row, tt0, tn, N, tid);
    st.store(sB, nullptr, tid);
    __syncthreads();

    if (active) {
      const int ng = (tn + kGroup - 1) / kGroup;
      for (int gi = ng - 1; gi >= 0; --gi) {
        const int g = gi * kGroup;
        const int64_t t = tt0 + g;
        const int nv = min(kGroup, tn - g);
        f2 u2[4], x2[4];
        if (a.vec && nv == kGroup) {
          const typename L::Raw8 ru = L::load8(a.u, row + t), rd = L::load8(a.delta, row + t);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            u2[p] = L::pair(ru, p);
            x2[p] = L::pair(rd, p);
          }
        } else {
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int j0 = 2 * p, j1 = 2 * p + 1;
            u2[p] = pk(j0 < nv ? L::one(a.u, row + t + j0) : 0.f, j1 < nv ? L::one(a.u, row + t + j1) : 0.f);
            x2[p] = pk(j0 < nv ? L::one(a.delta, row + t + j0) : 0.f, j1 < nv ? L::one(a.delta, row + t + j1) : 0.f);
          }
        }
        f2 dt2[4], du2[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const f2 x = add2(x2[p], bias2);
          dt2[p] = a.softplus ? softplus2(x) : x;
          du2[p] = mul2(dt2[p], u2[p]);
        }
#pragma unroll
        for (int j = kGroup - 1; j >= 0; --j) {
          if (j < nv) {
            const float dt = (j & 1) ? hi(dt2[j >> 1]) : lo(dt2[j >> 1]);
            const float du = (j & 1) ? hi(du2[j >> 1]) : lo(du2[j >> 1]);
            const f2 Rp = pk(R, R), dup = pk(du, du);
            const float* rb = sB + (g + j) * T::kRow;
#pragma unroll
            for (int q = 0; q < NP; q += 2) {
              const float4 bv = *reinterpret_cast<const float4*>(rb + 2 * q);
              if (live & (1u << q))
                acc[q] = fma2(ex2x2(mul2(Rp, A2[q])), mul2(dup, pk(bv.x, bv.y)), acc[q]);
              if (live & (2u << q))
                acc[q + 1] = fma2(ex2x2(mul2(Rp, A2[q + 1])), mul2(dup, pk(bv.z, bv.w)), acc[q + 1]);
            }
            R += dt;
          }
        }
      }
    }
    __syncthreads();
  }

  if (!active) return;
  a.ws_S[bd * a.nchunks + k] = R;
  float* H = a.ws_H + (bd * a.nchunks + k) * N;
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    if (2 * q < N) H[2 * q] = lo(acc[q]);
    if (2 * q + 1 < N) H[2 * q + 1] = hi(acc[q]);
  }
}

}  // namespace ssk
