// Full-sequence scan with one warp per channel: the lanes split time.
//
// Within a segment of 32 x kWT steps, lane l owns the kWT consecutive steps
// starting at l * kWT.  For every state pair the lane
//   1. computes its steps' decays e_t = exp(dt_t A) and input terms b_t = dt_t B_t u_t,
//      keeps them in registers and folds them into its zero-start end state;
//   2. joins a Kogge-Stone scan over the 32 lanes of the pairs
//      (decay product, end state) under (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2)
//      (the associative form of the recurrence; "Parallel scan", "Mamba: Linear-Time
//      Sequence Modeling with Selective State Spaces"), which gives the state entering
//      its first step from the state entering the segment;
//   3. runs the recurrence h = e h + b over its steps again from that state, with the
//      decays still in registers, and accumulates the readout C_t h_t.
// Each exp is computed once.  Segments follow one another in time; the state
// leaving a segment (that of lane 31) enters the next one.  A block is up to kWW warps
// (channels) of one batch row: the B and C rows of a segment, shared by those
// channels, are copied into shared memory by cp.async one segment ahead and
// widened to fp32 [pair][step] tiles once per block.
//
// Supported: the Euler or the zero-order-hold input weight, N <= 16, seqlen % 8 == 0,
// 16-byte aligned rows (u, delta, z, y, B, C).  Other shapes use the
// one-thread-per-channel kernels.
#include <algorithm>

#include "ss_device.cuh"
#include "ss_kernels.cuh"
#include "ss_launch.h"
#include "ss_occupancy.cuh"

namespace ssk {

namespace {

constexpr int kWT = 16;                 // steps per lane
constexpr int kWS = 32 * kWT;           // steps per segment
constexpr int kWW = 12;                 // most warps (channels) per block
constexpr int kWRow = kWS + kWS / kWT;  // tile row in f2 units: one pad slot per lane's steps

// Shared memory: B and C tiles (f2 [NP][kWRow] each), the raw B/C rows of the next
// segment ([B, C][NT][kWS] input elements), per warp A * log2(e), 1 / A (zero where
// A = 0) and the carried state as pairs, and per warp its channel's u, delta and z
// rows of a segment ([u, delta, z][kWS] input elements).
template <int NT, bool BF>
struct WarpLayout {
  static constexpr int NP = NT / 2;
  static constexpr int ES = BF ? 2 : 4;
  static constexpr int kTile = NP * kWRow * 8;
  static constexpr int oC = kTile;
  static constexpr int oRaw = 2 * kTile;
  static constexpr int kRaw = 2 * NT * kWS * ES;
  static constexpr int oA = oRaw + kRaw;
  static constexpr int oIA = oA + kWW * NP * 8;
  static constexpr int oH = oIA + kWW * NP * 8;
  static constexpr int oIn = oH + kWW * NP * 8;
  static constexpr int kIn = 3 * kWS * ES;
  static constexpr int kBytes = oIn + kWW * kIn;
};

// 16-byte asynchronous copy that reads src_bytes (16 or 0) and zero-fills the rest.
__device__ __forceinline__ void cp_async16_fill(unsigned sa, const void* gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ f2 shfl_up2(f2 v, int off) {
  return pk(__shfl_up_sync(0xffffffffu, lo(v), off), __shfl_up_sync(0xffffffffu, hi(v), off));
}

template <bool BF>
__device__ __forceinline__ float raw_elem(const unsigned char* p, int i) {
  if constexpr (BF) return bf16_lo(reinterpret_cast<const unsigned short*>(p)[i]);
  else return reinterpret_cast<const float*>(p)[i];
}

template <int NT, bool BF, bool HAS_Z, bool ZOH>
__global__ void __launch_bounds__(32 * kWW, 1) scan_warp_kernel(const ScanArgs a) {
  using L = In<BF>;
  using Lay = WarpLayout<NT, BF>;
  constexpr int NP = NT / 2;
  constexpr int ES = Lay::ES;
  extern __shared__ __align__(16) unsigned char sm[];
  f2* tB = reinterpret_cast<f2*>(sm);
  f2* tC = reinterpret_cast<f2*>(sm + Lay::oC);
  unsigned char* raw = sm + Lay::oRaw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  f2* sA = reinterpret_cast<f2*>(sm + Lay::oA) + warp * NP;
  f2* sIA = reinterpret_cast<f2*>(sm + Lay::oIA) + warp * NP;
  f2* sH = reinterpret_cast<f2*>(sm + Lay::oH) + warp * NP;
  unsigned char* sIn = sm + Lay::oIn + warp * Lay::kIn;   // [u, delta, z][kWS] of this warp's channel

  const int64_t b = blockIdx.y;
  const int ww = blockDim.x >> 5;        // warps (channels) in this block
  const int64_t d = (int64_t)blockIdx.x * ww + warp;
  const int N = (int)a.dstate;
  const int64_t Lsq = a.seqlen;
  // Debug build: the channel's rows, its A row, its state rows and the batch row of B and C.
  const bool active = d < a.dim && span_ok(a.err, (b * a.dim + d) * Lsq, Lsq, a.batch * a.dim * Lsq) &&
                      span_ok(a.err, d * N, N, a.dim * N) && span_ok(a.err, (b * a.dim + d) * N, N, a.batch * a.dim * N) &&
                      span_ok(a.err, b * N * Lsq, N * Lsq, a.batch * N * Lsq);
  const int64_t bd = b * a.dim + (active ? d : 0);
  const int64_t row = bd * Lsq;
  const int nseg = (int)((Lsq + kWS - 1) / kWS);

  if (lane < NP) {
    const int n0 = 2 * lane, n1 = 2 * lane + 1;
    float a0 = 0.f, a1 = 0.f, h0 = 0.f, h1 = 0.f;
    if (active) {
      if (n0 < N) a0 = a.A[d * N + n0];
      if (n1 < N) a1 = a.A[d * N + n1];
      if (a.h0) {
        if (n0 < N) h0 = a.h0[bd * N + n0];
        if (n1 < N) h1 = a.h0[bd * N + n1];
      }
    }
    sA[lane] = pk(a0 * kLog2e, a1 * kLog2e);
    sIA[lane] = pk(a0 != 0.f ? 1.f / a0 : 0.f, a1 != 0.f ? 1.f / a1 : 0.f);
    sH[lane] = pk(h0, h1);
  }
  const float bias = (a.delta_bias && active) ? a.delta_bias[d] : 0.f;
  const f2 bias2 = pk(bias, bias);
  const float Dd = (a.D && active) ? a.D[d] : 0.f;

  // Raw B and C rows of segment sg: [which][n][step], 16-byte chunks; chunks past
  // seqlen are zero-filled (seqlen % 8 == 0, so a chunk is wholly inside or outside).
  auto issue = [&](int sg) {
    constexpr int CPR = kWS * ES / 16;
    const int64_t t0 = (int64_t)sg * kWS;
    const int total = 2 * N * CPR;
    for (int c = threadIdx.x; c < total; c += blockDim.x) {
      const int which = c / (N * CPR);
      const int rem = c - which * N * CPR;
      const int n = rem / CPR, k = rem - n * CPR;
      const int64_t t = t0 + (int64_t)k * (16 / ES);
      const unsigned char* src =
          static_cast<const unsigned char*>(which ? a.C : a.B) + (b * N + n) * Lsq * ES;
      const bool ok = t < Lsq;
      cp_async16_fill(smem_addr(raw + ((which * NT + n) * kWS) * ES + k * 16), ok ? src + t * ES : src,
                      ok ? 16 : 0);
    }
    cp_async_commit();
  };
  // This warp's rows of arrays [first, first + count) (u, delta, z) for segment sg, by
  // its own lanes; chunks past seqlen are zero-filled.
  auto issue_in = [&](int sg, int first, int count) {
    constexpr int CPR = kWS * ES / 16;
    const int64_t t0 = (int64_t)sg * kWS;
    for (int arr = first; arr < first + count; ++arr) {
      const unsigned char* src =
          static_cast<const unsigned char*>(arr == 0 ? a.u : arr == 1 ? a.delta : a.z) + row * ES;
      for (int k = lane; k < CPR; k += 32) {
        const int64_t t = t0 + (int64_t)k * (16 / ES);
        const bool ok = t < Lsq;
        cp_async16_fill(smem_addr(sIn + arr * kWS * ES + k * 16), ok ? src + t * ES : src, ok ? 16 : 0);
      }
    }
    cp_async_commit();
  };
  // Widen the raw rows to the [pair][step] tiles; lane l's step i sits at l * (kWT + 1) + i.
  auto convert = [&]() {
    for (int u = threadIdx.x; u < NP * kWS; u += blockDim.x) {
      const int q = u / kWS, t = u - q * kWS;
      const int n0 = 2 * q, n1 = 2 * q + 1;
      const unsigned char* rB = raw;
      const unsigned char* rC = raw + NT * kWS * ES;
      const float b0 = n0 < N ? raw_elem<BF>(rB + n0 * kWS * ES, t) : 0.f;
      const float b1 = n1 < N ? raw_elem<BF>(rB + n1 * kWS * ES, t) : 0.f;
      const float c0 = n0 < N ? raw_elem<BF>(rC + n0 * kWS * ES, t) : 0.f;
      const float c1 = n1 < N ? raw_elem<BF>(rC + n1 * kWS * ES, t) : 0.f;
      const int o = q * kWRow + t + t / kWT;
      tB[o] = pk(b0, b1);
      tC[o] = pk(c0, c1);
    }
  };

  if (nseg > 0) {
    issue(0);
    if (active) issue_in(0, 0, HAS_Z ? 3 : 2);
  }
  for (int sg = 0; sg < nseg; ++sg) {
    cp_async_wait<0>();
    __syncthreads();  // rows of sg visible (B, C and each warp's inputs); tiles of sg - 1 done
    convert();
    __syncthreads();  // tiles of sg ready; the raw buffer is free
    if (sg + 1 < nseg) issue(sg + 1);
    if (!active) continue;

    const int64_t tb = (int64_t)sg * kWS + lane * kWT;
    const int64_t left = Lsq - tb;
    const int nv = left <= 0 ? 0 : (left >= kWT ? kWT : (int)left);  // a multiple of 8
    f2 dt2[kWT / 2], du2[kWT / 2], y2[kWT];
#pragma unroll
    for (int g = 0; g < kWT / 8; ++g) {
      if (8 * g < nv) {
        const unsigned off = (unsigned)((lane * kWT + 8 * g) * ES);
        const typename L::Raw8 ru = L::from_smem(smem_addr(sIn + off), 16);
        const typename L::Raw8 rd = L::from_smem(smem_addr(sIn + kWS * ES + off), 16);
        f2 dtg[4], dug[4];
        step_scalars<BF>(ru, rd, bias2, a.softplus, dtg, dug);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const f2 up = L::pair(ru, p);
          dt2[4 * g + p] = dtg[p];
          du2[4 * g + p] = ZOH ? up : dug[p];  // the hold weight multiplies u itself
          y2[8 * g + 2 * p] = pk(Dd * lo(up), 0.f);
          y2[8 * g + 2 * p + 1] = pk(Dd * hi(up), 0.f);
        }
      } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          dt2[4 * g + p] = pk(0.f, 0.f);
          du2[4 * g + p] = pk(0.f, 0.f);
          y2[8 * g + 2 * p] = pk(0.f, 0.f);
          y2[8 * g + 2 * p + 1] = pk(0.f, 0.f);
        }
      }
    }
    __syncwarp();  // every lane has read u and delta of sg: refill them with sg + 1
    if (sg + 1 < nseg) issue_in(sg + 1, 0, 2);
    f2 s2 = dt2[0];
#pragma unroll
    for (int p = 1; p < kWT / 2; ++p) s2 = add2(s2, dt2[p]);
    const float sdt = lo(s2) + hi(s2);

    // du2 holds dt * u (Euler) or u (zero-order hold).
    const f2* lB = tB + lane * (kWT + 1);
    const f2* lC = tC + lane * (kWT + 1);
#pragma unroll 1
    for (int q = 0; q < NP; ++q) {
      const f2 A2 = sA[q];
      const f2 iA = sIA[q];
      f2 e[kWT], bb[kWT];
      f2 agg = pk(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kWT; ++i) {
        const float dt = (i & 1) ? hi(dt2[i >> 1]) : lo(dt2[i >> 1]);
        const float du = (i & 1) ? hi(du2[i >> 1]) : lo(du2[i >> 1]);
        const f2 arg = mul2(pk(dt, dt), A2);
        e[i] = ex2x2(arg);
        if constexpr (ZOH) bb[i] = mul2(hold2(arg, e[i], pk(dt, dt), iA), mul2(pk(du, du), lB[q * kWRow + i]));
        else bb[i] = mul2(pk(du, du), lB[q * kWRow + i]);
        agg = fma2(e[i], agg, bb[i]);
      }
      // Inclusive scan over lanes of (decay product, zero-start end state).
      f2 ai = ex2x2(mul2(pk(sdt, sdt), A2)), bi = agg;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const f2 ap = shfl_up2(ai, off), bp = shfl_up2(bi, off);
        if (lane >= off) {
          bi = fma2(ai, bp, bi);
          ai = mul2(ai, ap);
        }
      }
      f2 ae = shfl_up2(ai, 1), be = shfl_up2(bi, 1);
      if (lane == 0) {
        ae = pk(1.f, 1.f);
        be = pk(0.f, 0.f);
      }
      f2 h = fma2(ae, sH[q], be);
#pragma unroll
      for (int i = 0; i < kWT; ++i) {
        h = fma2(e[i], h, bb[i]);
        y2[i] = fma2(lC[q * kWRow + i], h, y2[i]);
      }
      __syncwarp();
      if (lane == 31) sH[q] = h;  // steps past seqlen have e = 1, b = 0: h is the segment's end state
    }

    float yo[kWT];
#pragma unroll
    for (int i = 0; i < kWT; ++i) yo[i] = lo(y2[i]) + hi(y2[i]);
#pragma unroll
    for (int g = 0; g < kWT / 8; ++g) {
      if (8 * g < nv) {
        if constexpr (HAS_Z) {
          const typename L::Raw8 rz =
              L::from_smem(smem_addr(sIn + 2 * kWS * ES + (unsigned)((lane * kWT + 8 * g) * ES)), 16);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const f2 s = silu2(L::pair(rz, p));
            yo[8 * g + 2 * p] *= lo(s);
            yo[8 * g + 2 * p + 1] *= hi(s);
          }
        }
        float4* yp = reinterpret_cast<float4*>(a.y + row + tb + 8 * g);
        yp[0] = make_float4(yo[8 * g], yo[8 * g + 1], yo[8 * g + 2], yo[8 * g + 3]);
        yp[1] = make_float4(yo[8 * g + 4], yo[8 * g + 5], yo[8 * g + 6], yo[8 * g + 7]);
      }
    }
    if constexpr (HAS_Z) {
      __syncwarp();  // every lane has read z of sg
      if (sg + 1 < nseg) issue_in(sg + 1, 2, 1);
    }
  }

  if (active && a.last_state) {
    __syncwarp();
    if (lane < NP) {
      const f2 h = sH[lane];
      if (2 * lane < N) a.last_state[bd * N + 2 * lane] = lo(h);
      if (2 * lane + 1 < N) a.last_state[bd * N + 2 * lane + 1] = hi(h);
    }
  }
}

template <int NT, bool BF, bool HAS_Z, bool ZOH>
int go_warp(const ScanArgs& a, cudaStream_t s) {
  constexpr int bytes = WarpLayout<NT, BF>::kBytes;
  auto k = scan_warp_kernel<NT, BF, HAS_Z, ZOH>;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return (int)e;
  // Warps per block: 12, or fewer when there are too few channels to give every SM a
  // block, so that the channels spread over all SMs instead of sharing a few.
  DevInfo di;
  const int64_t sms = device_info(&di) && di.sms > 0 ? di.sms : 148;
  const int64_t ch = a.batch * a.dim;
  const int ww = (int)std::min<int64_t>(kWW, std::max<int64_t>(1, (ch + sms - 1) / sms));
  const dim3 grid((unsigned)((a.dim + ww - 1) / ww), (unsigned)a.batch);
  k<<<grid, 32 * ww, bytes, s>>>(a);
  return 0;
}

template <bool BF, bool HAS_Z, bool ZOH>
int dispatch_nt(const ScanArgs& a, cudaStream_t s) {
  if (a.dstate <= 4) return go_warp<4, BF, HAS_Z, ZOH>(a, s);
  if (a.dstate <= 8) return go_warp<8, BF, HAS_Z, ZOH>(a, s);
  return go_warp<16, BF, HAS_Z, ZOH>(a, s);
}

template <bool BF, bool HAS_Z>
int dispatch_warp(const ScanArgs& a, cudaStream_t s) {
  return a.zoh ? dispatch_nt<BF, HAS_Z, true>(a, s) : dispatch_nt<BF, HAS_Z, false>(a, s);
}

}  // namespace

bool warp_scan_available(const ScanArgs& a, bool bf16) {
  (void)bf16;
  return a.dstate >= 1 && a.dstate <= 16 && a.seqlen % 8 == 0 && a.vec && a.vec_bc;
}

int launch_scan_warp(const ScanArgs& a, bool bf16, bool has_z, cudaStream_t s) {
  if (bf16) return has_z ? dispatch_warp<true, true>(a, s) : dispatch_warp<true, false>(a, s);
  return has_z ? dispatch_warp<false, true>(a, s) : dispatch_warp<false, false>(a, s);
}

}  // namespace ssk
