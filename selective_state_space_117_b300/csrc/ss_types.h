// Argument blocks and launch constants shared by the host launchers and the kernels.
#pragma once

#include <cstdint>

namespace ssk {

constexpr int kCh = 64;        // channels (threads) per scan block

// Bits of the per-device status word that kernels write (atomicOr) instead of trapping.
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 1;   // a bounded wait on an asynchronous copy gave up
constexpr int kDevBounds = 2;    // a debug-build index check failed (SS_DEBUG_BOUNDS)
constexpr int kGroup = 8;      // time steps per vector load
constexpr int kDecodeThreads = 256;

enum Mode { kFull = 0, kLocal = 1, kFixup = 2 };

struct ScanArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  float* y;
  float* last_state;
  const float* h0;   // (batch, dim, N) initial state, or null for zeros
  float* ws_S;       // (nchunks, batch, dim): sum of dt over each chunk
  float* ws_H;       // (nchunks, batch, dim, N): chunk end state, then carry-in
  int64_t batch, dim, dstate, seqlen, chunk_len, nchunks;
  int ctiles;        // channel tiles (blocks) per (b, chunk)
  int softplus;
  int vec;           // 1: every row start is 16-byte aligned for u, delta, z and y
  int vec_bc;        // 1: every 8-step segment of a B or C row is 16-byte aligned
  int* err;          // device status word (bounded waits record a timeout here), may be null
  int zoh;           // 1: zero-order-hold input weight (exp(dt A) - 1) / A instead of dt
  int64_t local_chunks;  // the local pass covers chunks 0 .. local_chunks - 1
  int* perm;         // (dim) workspace for the channel order of the grouped local pass, or null
};

// Backward pass.  Chunks of kBwdChunk steps; the workspace holds, per (chunk k, b, d),
// chunk-major like the forward's:
//   ws_S[k]    sum of dt over the chunk (written by the forward local pass)
//   ws_H[k][n] the state entering chunk k (forward local pass, then the carry)
//   ws_G[k][n] the chunk's adjoint sum, then mu_k = exp(A dt_{t1}) lambda_{t1}: the
//              gradient reaching the chunk's last state from the steps after it
constexpr int kBwdChunk = 64;

struct BwdArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  const float* dy;       // (batch, dim, L) fp32
  const float* dlast;    // (batch, dim, N) or null
  float* du;             // (batch, dim, L)
  float* ddelta;         // (batch, dim, L)
  float* dz;             // (batch, dim, L) or null (only with z)
  float* dA;             // (dim, N), accumulated
  float* dB;             // (batch, N, L), accumulated
  float* dC;             // (batch, N, L), accumulated
  float* dD;             // (dim) or null, accumulated
  float* dbias;          // (dim) or null, accumulated
  float* dh0;            // (batch, dim, N) or null
  float* ws_S;
  float* ws_H;
  float* ws_G;
  int64_t batch, dim, dstate, seqlen, nchunks;
  int ctiles;            // channel tiles per (b, chunk) of the launched kernel
  int softplus;
  int vec;               // 1: u/delta/z rows, dy and the fp32 gradient rows allow 16-byte group loads
  int vec_bc;            // 1: B/C rows allow 16-byte loads of 8-step groups
  int zoh;               // 1: zero-order-hold input weight
  int* err;              // device status word (debug-build index checks record here), may be null
};

// Causal depthwise conv1d of width 4 over (rows = batch * dim, seqlen).
struct ConvArgs {
  const void* x;
  const float* w;      // (dim, 4), 16-byte aligned
  const float* bias;   // (dim) or null
  void* out;
  int64_t rows, dim, seqlen, nseg;
  int vec;             // 1: rows are 16-byte aligned for 8-element vectors
  int* err;            // device status word (debug-build index checks record here), may be null
};

// One decode step, one thread per (b, d).
struct DecodeArgs {
  float* state;
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  float* y;
  int64_t batch, dim, dstate;
  int softplus;
  int vec;           // 1: N % 4 == 0 and state, A, B, C rows allow 16/8-byte vector access
  int zoh;           // 1: zero-order-hold input weight
  int* err;          // device status word (a bounded wait records a timeout here), may be null
};

}  // namespace ssk
