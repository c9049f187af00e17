// C ABI of the selective scan library: argument validation on the host, then
// kernel launches on the caller's stream.  See include/ss_scan.h for the
// contract of every entry point.
#include <cstdint>
#include <mutex>
#include <unordered_map>

#include <cuda_runtime.h>

#include "ss_launch.h"
#include "ss_scan.h"

namespace {

thread_local int g_last_cuda = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda = (int)e;
  return SS_ECUDA;
}

// After enqueueing kernels: report launch errors (non-sticky errors are cleared).
int launched() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SS_OK : cuda_fail(e);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t in_size(int32_t dtype) { return dtype == SS_BF16 ? 2 : 4; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int64_t kMaxGridX = 2147483647;
constexpr int64_t kMaxGridY = 65535;
constexpr size_t kWsAlign = 256;
// ss_scan_fwd takes the one-warp-per-channel schedule below this many channels (batch * dim):
// Euler input weight, and the zero-order hold (whose weight slows the one-thread-per-channel
// kernel about 2.9x but the warp kernel only about 1.4x).
constexpr int64_t kWarpBelowChannels = 9216;
constexpr int64_t kWarpBelowChannelsZoh = 20480;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Device address of one of this library's __device__ variables on the current device.
// The address belongs to the device's current context: after cudaDeviceReset the next
// context loads the module afresh, possibly elsewhere, so a cached address may be stale.
// The address is therefore looked up again (a host-side table query) on every call whose
// stream is not being captured, and the last address seen on each device is kept for
// calls made during a capture, where a lookup that had to load the module would not be
// allowed.  Returns nullptr (and the CUDA error in *err) when the lookup fails.
constexpr int kMaxDevices = 256;

struct SymbolCache {
  std::mutex mu;
  void* ptr[kMaxDevices] = {};
};

void* symbol_on_device(SymbolCache& c, const void* symbol, cudaStream_t s, cudaError_t* err) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *err = e; return nullptr; }
  if (dev < 0 || dev >= kMaxDevices) { *err = cudaErrorInvalidDevice; return nullptr; }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone;
  if (capturing) (void)cudaGetLastError();   // a refused query leaves a (non-sticky) error behind
  std::lock_guard<std::mutex> lock(c.mu);
  if (!capturing || c.ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess) { *err = e; return nullptr; }
    c.ptr[dev] = p;
  }
  return c.ptr[dev];
}

// The device status word: kernels whose bounded waits give up record it here.
__device__ int g_dev_status;
SymbolCache g_status_cache;

// The word's address for the kernels about to be launched on stream s, or nullptr (the
// kernels then skip recording a timeout; the CUDA error is left in *err when given).
int* device_status_word(cudaStream_t s, cudaError_t* err = nullptr) {
  cudaError_t e = cudaSuccess;
  void* p = symbol_on_device(g_status_cache, (const void*)&g_dev_status, s, &e);
  if (err) *err = e;
  return static_cast<int*>(p);
}

// Shape, dtype and pointer checks shared by the two full-sequence entry points.
int check_scan(const ss_dims* dims, const void* u, const void* delta, const float* A, const void* B,
               const void* C, const float* D, const void* z, const float* delta_bias, const float* y,
               const float* last_state, int32_t allowed_flags = SS_FLAG_ZOH) {
  if (!dims) return SS_EINVAL;
  const ss_dims& d = *dims;
  if (d.in_dtype != SS_F32 && d.in_dtype != SS_BF16) return SS_EDTYPE;
  if (d.batch < 0 || d.dim < 0 || d.dstate < 0 || d.seqlen < 0) return SS_EINVAL;
  if ((d.flags & ~allowed_flags) != 0) return SS_EINVAL;
  if ((d.flags & SS_FLAG_SCHED_THREAD) && (d.flags & SS_FLAG_SCHED_WARP)) return SS_EINVAL;
  if (d.dstate > SS_MAX_DSTATE || d.batch > kMaxGridY) return SS_EINVAL;
  if (ceil_div(d.dim, ssk::kCh) > kMaxGridX) return SS_EINVAL;
  const size_t es = in_size(d.in_dtype);
  const bool rows = d.batch > 0 && d.dim > 0 && d.seqlen > 0;
  if (rows && (!u || !delta || !y)) return SS_EINVAL;
  if (rows && d.dstate > 0 && (!B || !C || !A)) return SS_EINVAL;
  if (!aligned(u, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) || !aligned(z, es))
    return SS_EALIGN;
  if (!aligned(A, 4) || !aligned(D, 4) || !aligned(delta_bias, 4) || !aligned(y, 4) || !aligned(last_state, 4))
    return SS_EALIGN;
  return SS_OK;
}

ssk::ScanArgs make_scan_args(const ss_dims& d, const void* u, const void* delta, const float* A, const void* B,
                             const void* C, const float* D, const void* z, const float* delta_bias,
                             int softplus_flag, float* y, float* last_state, int64_t chunk_len,
                             cudaStream_t s) {
  ssk::ScanArgs a{};
  a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.delta_bias = delta_bias;
  a.y = y; a.last_state = last_state;
  a.batch = d.batch; a.dim = d.dim; a.dstate = d.dstate; a.seqlen = d.seqlen;
  a.chunk_len = chunk_len;
  a.nchunks = ceil_div(d.seqlen, chunk_len);
  a.ctiles = (int)ceil_div(d.dim, ssk::kCh);
  a.softplus = softplus_flag ? 1 : 0;
  // 16-byte vector loads along a row need every row start and every group start aligned.
  const size_t es = in_size(d.in_dtype);
  const bool rows16 = (d.seqlen * (int64_t)es) % 16 == 0 && (d.seqlen * 4) % 16 == 0;
  const bool ptr16 = aligned(u, 16) && aligned(delta, 16) && aligned(z, 16) && aligned(y, 16);
  a.vec = (rows16 && ptr16 && chunk_len % ssk::kGroup == 0) ? 1 : 0;
  // B/C rows are staged in 8-step segments from tile starts that are multiples of 8 steps.
  const bool bc16 = (d.seqlen * (int64_t)es) % 16 == 0 && aligned(B, 16) && aligned(C, 16);
  a.vec_bc = (bc16 && chunk_len % ssk::kGroup == 0) ? 1 : 0;
  a.err = device_status_word(s);
  a.zoh = (d.flags & SS_FLAG_ZOH) ? 1 : 0;
  return a;
}

// The final state when there is nothing to scan (L = 0): the initial state, i.e.
// zeros or a copy of h0.
int initial_state(const ss_dims& d, const float* h0, float* last_state, cudaStream_t s) {
  if (!last_state) return SS_OK;
  const size_t n = (size_t)(d.batch * d.dim * d.dstate);
  if (n == 0) return SS_OK;
  const cudaError_t e = h0 ? cudaMemcpyAsync(last_state, h0, n * sizeof(float), cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(last_state, 0, n * sizeof(float), s);
  return e == cudaSuccess ? SS_OK : cuda_fail(e);
}

int scan_fwd_impl(const ss_dims* dims, const float* h0, const void* u, const void* delta, const float* A,
                  const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                  int softplus_flag, float* y, float* last_state, cudaStream_t s) {
  const int st = check_scan(dims, u, delta, A, B, C, D, z, delta_bias, y, last_state,
                            SS_FLAG_ZOH | SS_FLAG_SCHED_THREAD | SS_FLAG_SCHED_WARP);
  if (st != SS_OK) return st;
  if (!aligned(h0, 4)) return SS_EALIGN;
  const ss_dims& d = *dims;
  if (d.batch == 0 || d.dim == 0) return SS_OK;
  if (d.seqlen == 0) return initial_state(d, h0, last_state, s);
  ssk::ScanArgs a = make_scan_args(d, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state,
                                   d.seqlen, s);
  a.h0 = h0;
  const dim3 grid((unsigned)a.ctiles, (unsigned)d.batch);
  const bool bf = d.in_dtype == SS_BF16;
  // Schedule.  One thread per channel advances a channel by about one step per 110 ns
  // (Euler; 290 ns with the hold weight) while the GPU is far from full, and one warp per
  // channel moves about 90 G elements/s (73 G with the hold weight; B300, N = 16): the two
  // meet near 10 K channels (21 K with the hold weight), whatever L is.
  const bool warp_ok = ssk::warp_scan_available(a, bf);
  if (d.flags & SS_FLAG_SCHED_WARP) {
    if (!warp_ok) return SS_EINVAL;
  }
  const int64_t below = a.zoh ? kWarpBelowChannelsZoh : kWarpBelowChannels;
  const bool use_warp = (d.flags & SS_FLAG_SCHED_WARP) ||
                        (!(d.flags & SS_FLAG_SCHED_THREAD) && warp_ok && d.batch * d.dim < below);
  if (use_warp) {
    const int rc = ssk::launch_scan_warp(a, bf, z != nullptr, s);
    if (rc != 0) return cuda_fail((cudaError_t)rc);
    return launched();
  }
  if (ssk::tma_available(a, bf, ssk::kFull) && ssk::launch_scan_tma(a, bf, z != nullptr, ssk::kFull, grid, s) == 0)
    return launched();
  if (ssk::launch_scan_full(a, bf, z != nullptr, grid, s) != 0) return SS_EINVAL;
  return launched();
}

}  // namespace

extern "C" {

int ss_scan_fwd(const ss_dims* dims, const void* u, const void* delta, const float* A, const void* B,
                const void* C, const float* D, const void* z, const float* delta_bias, int softplus_flag,
                float* y, float* last_state, ss_stream_t stream) {
  return scan_fwd_impl(dims, nullptr, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state,
                       reinterpret_cast<cudaStream_t>(stream));
}

int ss_scan_fwd_h0(const ss_dims* dims, const float* h0, const void* u, const void* delta, const float* A,
                   const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                   int softplus_flag, float* y, float* last_state, ss_stream_t stream) {
  return scan_fwd_impl(dims, h0, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state,
                       reinterpret_cast<cudaStream_t>(stream));
}

// The chunked workspace: S (K, batch, dim) fp32, then H (K, batch, dim, N) fp32, then the
// channel order of the grouped local pass (dim) int32, each part 256-byte aligned.
struct ChunkedWs {
  size_t s_off, h_off, perm_off, bytes;
};

ChunkedWs chunked_ws_layout(const ss_dims& d, int64_t chunk_len) {
  const int64_t K = ceil_div(d.seqlen, chunk_len);
  ChunkedWs w;
  w.s_off = 0;
  w.h_off = align_up((size_t)(d.batch * d.dim * K) * sizeof(float), kWsAlign);
  w.perm_off = w.h_off + align_up((size_t)(d.batch * d.dim * K * d.dstate) * sizeof(float), kWsAlign);
  w.bytes = w.perm_off + (size_t)d.dim * sizeof(int);
  return w;
}

size_t ss_scan_chunked_workspace_bytes(const ss_dims* dims, int64_t chunk_len) {
  if (!dims || chunk_len < 1 || dims->batch < 0 || dims->dim < 0 || dims->dstate < 0 || dims->seqlen < 0)
    return 0;
  return chunked_ws_layout(*dims, chunk_len).bytes;
}

}  // extern "C"

namespace {

int chunked_phase_impl(int phase, const ss_dims* dims, const float* h0, const void* u, const void* delta,
                       const float* A, const void* B, const void* C, const float* D, const void* z,
                       const float* delta_bias, int softplus_flag, float* y, float* last_state, int64_t chunk_len,
                       void* workspace, size_t workspace_bytes, cudaStream_t s) {
  if (phase < SS_PHASE_LOCAL || phase > SS_PHASE_FIXUP) return SS_EINVAL;
  const int st = check_scan(dims, u, delta, A, B, C, D, z, delta_bias, y, last_state);
  if (st != SS_OK) return st;
  if (!aligned(h0, 4)) return SS_EALIGN;
  if (chunk_len < 1) return SS_EINVAL;
  const ss_dims& d = *dims;
  if (d.batch == 0 || d.dim == 0) return SS_OK;
  if (d.seqlen == 0) return phase == SS_PHASE_CARRY ? initial_state(d, h0, last_state, s) : SS_OK;
  const size_t need = ss_scan_chunked_workspace_bytes(dims, chunk_len);
  if (!workspace || !aligned(workspace, kWsAlign) || workspace_bytes < need) return SS_EWORKSPACE;
  ssk::ScanArgs a = make_scan_args(d, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state,
                                   chunk_len, s);
  a.h0 = h0;
  if ((int64_t)a.ctiles * a.nchunks > kMaxGridX) return SS_EINVAL;
  const ChunkedWs lay = chunked_ws_layout(d, chunk_len);
  char* ws = static_cast<char*>(workspace);
  a.ws_S = reinterpret_cast<float*>(ws + lay.s_off);
  a.ws_H = reinterpret_cast<float*>(ws + lay.h_off);
  a.perm = reinterpret_cast<int*>(ws + lay.perm_off);
  // The local pass leaves out the last chunk: only the carry into each chunk is needed from it,
  // and the final state comes out of the last chunk's fix-up.
  a.local_chunks = a.nchunks - 1;
  const dim3 grid((unsigned)(a.ctiles * a.nchunks), (unsigned)d.batch);
  const bool bf = d.in_dtype == SS_BF16;
  int rc = 0;
  if (phase == SS_PHASE_LOCAL) {
    const dim3 lgrid((unsigned)(a.ctiles * a.local_chunks), (unsigned)d.batch);
    if (a.local_chunks == 0) {
      rc = 0;
    } else if (softplus_flag && ssk::local_sorted_available(a, bf)) {
      rc = ssk::launch_local_sorted(a, bf, s);
    } else if (!(ssk::tma_available(a, bf, ssk::kLocal) && ssk::launch_local_tma(a, bf, lgrid, s) == 0)) {
      rc = ssk::launch_scan_local(a, bf, lgrid, s);
    }
  } else if (phase == SS_PHASE_CARRY) {
    rc = ssk::launch_carry(a, s);
  } else if (!(ssk::tma_available(a, bf, ssk::kFixup) &&
               ssk::launch_scan_tma(a, bf, z != nullptr, ssk::kFixup, grid, s) == 0)) {
    rc = ssk::launch_scan_fixup(a, bf, z != nullptr, grid, s);
  }
  if (rc != 0) return SS_EINVAL;
  return launched();
}

int chunked_impl(const ss_dims* dims, const float* h0, const void* u, const void* delta, const float* A,
                 const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                 int softplus_flag, float* y, float* last_state, int64_t chunk_len, void* workspace,
                 size_t workspace_bytes, cudaStream_t s) {
  for (int phase = SS_PHASE_LOCAL; phase <= SS_PHASE_FIXUP; ++phase) {
    const int st = chunked_phase_impl(phase, dims, h0, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y,
                                      last_state, chunk_len, workspace, workspace_bytes, s);
    if (st != SS_OK) return st;
  }
  return SS_OK;
}

// Alternates, per state array, the order in which a decode step takes the state's ranges
// (see launch_decode).  Only the order changes, never a result; a step captured into a CUDA
// graph keeps the order it was captured with, so consecutive captured steps alternate too.
int decode_reverse(const float* state) {
  static std::mutex mu;
  static std::unordered_map<const float*, unsigned> steps;
  std::lock_guard<std::mutex> lock(mu);
  if (steps.size() > 4096) steps.clear();   // bound the table; an order reset only costs L2 hits
  return (int)(steps[state]++ & 1u);
}

}  // namespace

extern "C" {

int ss_scan_chunked_phase(int phase, const ss_dims* dims, const void* u, const void* delta, const float* A,
                          const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                          int softplus_flag, float* y, float* last_state, int64_t chunk_len, void* workspace,
                          size_t workspace_bytes, ss_stream_t stream) {
  return chunked_phase_impl(phase, dims, nullptr, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y,
                            last_state, chunk_len, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int ss_scan_chunked(const ss_dims* dims, const void* u, const void* delta, const float* A, const void* B,
                    const void* C, const float* D, const void* z, const float* delta_bias, int softplus_flag,
                    float* y, float* last_state, int64_t chunk_len, void* workspace, size_t workspace_bytes,
                    ss_stream_t stream) {
  return chunked_impl(dims, nullptr, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, chunk_len,
                      workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int ss_scan_chunked_h0(const ss_dims* dims, const float* h0, const void* u, const void* delta, const float* A,
                       const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                       int softplus_flag, float* y, float* last_state, int64_t chunk_len, void* workspace,
                       size_t workspace_bytes, ss_stream_t stream) {
  return chunked_impl(dims, h0, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, chunk_len,
                      workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int ss_state_update(const ss_dims* dims, float* state, const void* u, const void* delta, const float* A,
                    const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                    int softplus_flag, float* y, ss_stream_t stream) {
  if (!dims) return SS_EINVAL;
  const ss_dims& d = *dims;
  if (d.in_dtype != SS_F32 && d.in_dtype != SS_BF16) return SS_EDTYPE;
  if (d.batch < 0 || d.dim < 0 || d.dstate < 0 || d.dstate > SS_MAX_DSTATE || d.batch > kMaxGridY)
    return SS_EINVAL;
  if ((d.flags & ~SS_FLAG_ZOH) != 0) return SS_EINVAL;
  if (ceil_div(d.dim, ssk::kCh) > kMaxGridX) return SS_EINVAL;
  if (d.batch == 0 || d.dim == 0) return SS_OK;
  if (!u || !delta || !y) return SS_EINVAL;
  if (d.dstate > 0 && (!state || !A || !B || !C)) return SS_EINVAL;
  const size_t es = in_size(d.in_dtype);
  if (!aligned(u, es) || !aligned(delta, es) || !aligned(B, es) || !aligned(C, es) || !aligned(z, es))
    return SS_EALIGN;
  if (!aligned(state, 4) || !aligned(A, 4) || !aligned(D, 4) || !aligned(delta_bias, 4) || !aligned(y, 4))
    return SS_EALIGN;
  ssk::DecodeArgs a{};
  a.state = state; a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z;
  a.delta_bias = delta_bias; a.y = y;
  a.batch = d.batch; a.dim = d.dim; a.dstate = d.dstate;
  a.softplus = softplus_flag ? 1 : 0;
  a.zoh = (d.flags & SS_FLAG_ZOH) ? 1 : 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  a.err = device_status_word(s);
  const uintptr_t bc_align = d.in_dtype == SS_BF16 ? 8 : 16;
  a.vec = (d.dstate % 4 == 0 && aligned(state, 16) && aligned(A, 16) && aligned(B, bc_align) && aligned(C, bc_align))
              ? 1 : 0;
  if (d.dim > (int64_t)INT32_MAX / 16) return SS_EINVAL;   // (channel, lane) index of a batch row fits int
  if (ssk::launch_decode(a, d.in_dtype == SS_BF16, z != nullptr, decode_reverse(state), s) != 0) return SS_EINVAL;
  return launched();
}

int ss_causal_conv1d(const ss_dims* dims, const void* x, const float* weight, const float* bias, int silu_flag,
                     void* out, ss_stream_t stream) {
  if (!dims) return SS_EINVAL;
  const ss_dims& d = *dims;
  if (d.in_dtype != SS_F32 && d.in_dtype != SS_BF16) return SS_EDTYPE;
  if (d.batch < 0 || d.dim < 0 || d.seqlen < 0) return SS_EINVAL;
  if (d.flags != 0) return SS_EINVAL;   // no input weight or schedule to choose
  if (d.batch == 0 || d.dim == 0 || d.seqlen == 0) return SS_OK;
  if (!x || !weight || !out) return SS_EINVAL;
  const size_t es = in_size(d.in_dtype);
  if (!aligned(x, es) || !aligned(out, es) || !aligned(weight, 16) || !aligned(bias, 4)) return SS_EALIGN;
  ssk::ConvArgs a{};
  a.x = x; a.w = weight; a.bias = bias; a.out = out;
  a.rows = d.batch * d.dim; a.dim = d.dim; a.seqlen = d.seqlen;
  a.nseg = ssk::conv1d_segments(d.seqlen);
  a.err = device_status_word(reinterpret_cast<cudaStream_t>(stream));
  a.vec = ((d.seqlen * (int64_t)es) % 16 == 0 && aligned(x, 16) && aligned(out, 16)) ? 1 : 0;
  if (ssk::launch_conv1d(a, d.in_dtype == SS_BF16, silu_flag != 0, reinterpret_cast<cudaStream_t>(stream)) != 0)
    return SS_EINVAL;
  return launched();
}

size_t ss_scan_bwd_workspace_bytes(const ss_dims* dims) {
  if (!dims || dims->batch < 0 || dims->dim < 0 || dims->dstate < 0 || dims->seqlen < 0) return 0;
  const int64_t K = ceil_div(dims->seqlen, ssk::kBwdChunk);
  const size_t s_bytes = (size_t)(dims->batch * dims->dim * K) * sizeof(float);
  const size_t h_bytes = (size_t)(dims->batch * dims->dim * K * dims->dstate) * sizeof(float);
  return align_up(s_bytes, kWsAlign) + align_up(h_bytes, kWsAlign) + h_bytes;
}

int ss_scan_bwd(const ss_dims* dims, const float* h0, const void* u, const void* delta, const float* A,
                const void* B, const void* C, const float* D, const void* z, const float* delta_bias,
                int softplus_flag, const float* dy, const float* dlast_state, float* du, float* ddelta, float* dA,
                float* dB, float* dC, float* dD, float* dz, float* ddelta_bias, float* dh0, void* workspace,
                size_t workspace_bytes, ss_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int st = check_scan(dims, u, delta, A, B, C, D, z, delta_bias, dy, nullptr);
  if (st != SS_OK) return st;
  const ss_dims& d = *dims;

  const bool rows = d.batch > 0 && d.dim > 0 && d.seqlen > 0;
  if (rows && (!du || !ddelta)) return SS_EINVAL;
  if (rows && d.dstate > 0 && (!dB || !dC)) return SS_EINVAL;
  if (d.dim > 0 && d.dstate > 0 && !dA) return SS_EINVAL;
  if (dz && !z) return SS_EINVAL;
  for (const void* p : {(const void*)h0, (const void*)dlast_state, (const void*)du, (const void*)ddelta,
                        (const void*)dA, (const void*)dB, (const void*)dC, (const void*)dD, (const void*)dz,
                        (const void*)ddelta_bias, (const void*)dh0})
    if (!aligned(p, 4)) return SS_EALIGN;
  const bool work = d.batch > 0 && d.dim > 0 && d.seqlen > 0;
  const size_t need = ss_scan_bwd_workspace_bytes(dims);
  if (work && (!workspace || !aligned(workspace, kWsAlign) || workspace_bytes < need)) return SS_EWORKSPACE;
  if (work && (int64_t)ceil_div(d.dim, ssk::kCh) * ceil_div(d.seqlen, ssk::kBwdChunk) > kMaxGridX) return SS_EINVAL;
  if (work && (int64_t)ssk::bwd_main_ctiles(d.dim, d.dstate) * ceil_div(d.seqlen, ssk::kBwdChunk) > kMaxGridX)
    return SS_EINVAL;

  // Accumulated gradients start from zero.
  auto zero = [&](float* p, int64_t n) -> int {
    if (!p || n <= 0) return SS_OK;
    const cudaError_t e = cudaMemsetAsync(p, 0, (size_t)n * sizeof(float), s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e);
  };
  int rc = SS_OK;
  if ((rc = zero(dA, d.dim * d.dstate)) != SS_OK || (rc = zero(dB, d.batch * d.dstate * d.seqlen)) != SS_OK ||
      (rc = zero(dC, d.batch * d.dstate * d.seqlen)) != SS_OK || (rc = zero(dD, d.dim)) != SS_OK ||
      (rc = zero(ddelta_bias, d.dim)) != SS_OK)
    return rc;
  if (d.batch == 0 || d.dim == 0) return SS_OK;
  if (d.seqlen == 0) {                                      // dh0 = dlast
    if (!dh0) return SS_OK;
    const size_t n = (size_t)(d.batch * d.dim * d.dstate) * sizeof(float);
    if (n == 0) return SS_OK;
    const cudaError_t e = dlast_state ? cudaMemcpyAsync(dh0, dlast_state, n, cudaMemcpyDeviceToDevice, s)
                                      : cudaMemsetAsync(dh0, 0, n, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e);
  }

  // Workspace: the chunks' dt sums, forward end states (then the states entering them) and
  // adjoint sums (then the gradients leaving them), at the backward's chunk length.
  ssk::ScanArgs f = make_scan_args(d, u, delta, A, B, C, D, z, delta_bias, softplus_flag, nullptr, nullptr,
                                   ssk::kBwdChunk, s);
  f.h0 = h0;
  const int64_t K = f.nchunks;
  f.local_chunks = K;   // the carry combines every chunk the local passes covered
  char* ws = static_cast<char*>(workspace);
  const size_t s_bytes = align_up((size_t)(d.batch * d.dim * K) * sizeof(float), kWsAlign);
  const size_t h_bytes = align_up((size_t)(d.batch * d.dim * K * d.dstate) * sizeof(float), kWsAlign);
  f.ws_S = reinterpret_cast<float*>(ws);
  f.ws_H = reinterpret_cast<float*>(ws + s_bytes);
  const bool bf = d.in_dtype == SS_BF16;

  ssk::BwdArgs a{};
  a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.delta_bias = delta_bias;
  a.dy = dy; a.dlast = dlast_state;
  a.du = du; a.ddelta = ddelta; a.dz = dz; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dbias = ddelta_bias;
  a.dh0 = dh0;
  a.ws_S = f.ws_S; a.ws_H = f.ws_H;
  a.ws_G = reinterpret_cast<float*>(ws + s_bytes + h_bytes);
  a.batch = d.batch; a.dim = d.dim; a.dstate = d.dstate; a.seqlen = d.seqlen; a.nchunks = K;
  a.softplus = softplus_flag ? 1 : 0;
  a.zoh = (d.flags & SS_FLAG_ZOH) ? 1 : 0;
  a.err = f.err;
  const size_t es = in_size(d.in_dtype);
  const bool rows16 = (d.seqlen * (int64_t)es) % 16 == 0 && (d.seqlen * 4) % 16 == 0;
  a.vec = (rows16 && aligned(u, 16) && aligned(delta, 16) && aligned(z, 16) && aligned(dy, 16) && aligned(du, 16) &&
           aligned(ddelta, 16) && aligned(dz, 16) && aligned(dB, 8) && aligned(dC, 8)) ? 1 : 0;
  a.vec_bc = ((d.seqlen * (int64_t)es) % 16 == 0 && aligned(B, 16) && aligned(C, 16)) ? 1 : 0;
  if (ssk::launch_bwd_locals(a, bf, z != nullptr, s) != 0) return SS_EINVAL;
  if (ssk::launch_carry(f, s) != 0) return SS_EINVAL;
  const int lrc = ssk::launch_bwd(a, bf, z != nullptr, s);
  if (lrc < 0) return SS_EINVAL;                             // unsupported dstate (caught above)
  if (lrc > 0) return cuda_fail(cudaGetLastError());         // the kernel attribute could not be set
  return launched();
}

const char* ss_status_string(int status) {
  switch (status) {
    case SS_OK: return "SS_OK";
    case SS_EINVAL: return "SS_EINVAL: invalid size or missing required pointer";
    case SS_EALIGN: return "SS_EALIGN: pointer not aligned to its element size";
    case SS_EDTYPE: return "SS_EDTYPE: unsupported input dtype";
    case SS_EWORKSPACE: return "SS_EWORKSPACE: workspace missing, misaligned or too small";
    case SS_ECUDA: return "SS_ECUDA: CUDA launch or call failed";
    case SS_ETIMEOUT: return "SS_ETIMEOUT: a bounded device wait ran out";
    case SS_EBOUNDS: return "SS_EBOUNDS: a device-side index check failed (debug build)";
    default: return "unknown ss_status";
  }
}

int ss_last_cuda_error(void) { return g_last_cuda; }

int ss_selftest_wait_timeout(ss_stream_t stream) {
  cudaError_t e = cudaSuccess;
  int* word = device_status_word(reinterpret_cast<cudaStream_t>(stream), &e);
  if (!word) return cuda_fail(e);
  ssk::launch_wait_timeout(word, reinterpret_cast<cudaStream_t>(stream));
  return launched();
}

int ss_measure_ex2(int64_t blocks, int iters, float* sink, uint64_t* ex2_count, ss_stream_t stream) {
  if (blocks < 1 || blocks > kMaxGridX || iters < 1 || !sink || !ex2_count) return SS_EINVAL;
  if (!aligned(sink, 4)) return SS_EALIGN;
  *ex2_count = (uint64_t)blocks * ssk::kEx2Threads * ssk::kEx2Chains * (uint64_t)iters;
  ssk::launch_ex2_rate(blocks, iters, sink, reinterpret_cast<cudaStream_t>(stream));
  return launched();
}

int ss_device_status(int clear) {
  cudaError_t e = cudaSuccess;
  int* word = device_status_word(nullptr, &e);
  if (!word) return cuda_fail(e);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  int v = 0;
  e = cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (clear && v != 0) {
    e = cudaMemset(word, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (v & ssk::kDevBounds) return SS_EBOUNDS;
  return v == 0 ? SS_OK : SS_ETIMEOUT;
}

int ss_selftest_bounds(ss_stream_t stream) {
  cudaError_t e = cudaSuccess;
  int* word = device_status_word(reinterpret_cast<cudaStream_t>(stream), &e);
  if (!word) return cuda_fail(e);
  ssk::launch_bounds_check(word, reinterpret_cast<cudaStream_t>(stream));
  return launched();
}

int ss_debug_bounds_build(void) {
#ifdef SS_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

}  // extern "C"

// ---------------------------------------------------------------------------
// ss_scan_chunked_static: the chunked scan on a workspace that the library owns.
//
// The workspace is one file-scope __device__ array of SS_STATIC_WORKSPACE_BYTES.
// In host code the name g_static_ws is only a host-side handle for the symbol,
// not a device address, so it is never passed to a kernel; its device address
// is looked up with cudaGetSymbolAddress (with the device current) by
// symbol_on_device above: on every call made outside a stream capture, and
// from the last lookup on that device during a capture.
namespace {

__device__ __align__(256) unsigned char g_static_ws[SS_STATIC_WORKSPACE_BYTES];
SymbolCache g_static_cache;

}  // namespace

extern "C" int ss_scan_chunked_static(const ss_dims* dims, const void* u, const void* delta, const float* A,
                                      const void* B, const void* C, const float* D, const void* z,
                                      const float* delta_bias, int softplus_flag, float* y, float* last_state,
                                      int64_t chunk_len, ss_stream_t stream) {
  if (!dims || chunk_len < 1) return SS_EINVAL;
  // Reject problems whose workspace does not fit before touching the device.
  if (ss_scan_chunked_workspace_bytes(dims, chunk_len) > (size_t)SS_STATIC_WORKSPACE_BYTES) return SS_EWORKSPACE;
  cudaError_t e = cudaSuccess;
  void* ws = symbol_on_device(g_static_cache, (const void*)&g_static_ws, reinterpret_cast<cudaStream_t>(stream), &e);
  if (!ws) return cuda_fail(e);
  // The chunked phases write every workspace entry before reading it, so the
  // previous call's contents need no clearing.
  return ss_scan_chunked(dims, u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, chunk_len, ws,
                         (size_t)SS_STATIC_WORKSPACE_BYTES, stream);
}
