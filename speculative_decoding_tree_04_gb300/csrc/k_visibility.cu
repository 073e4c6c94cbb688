// k_visibility.cu -- draft-tree ancestor-or-self bitsets (tv_build_visibility).
//
// "The Precision Imperative: Validating Numerical Accuracy in a Custom CUDA Attention
// Kernel", §Context: the verify kernel masks which tree tokens each query may see; here a
// node sees its ancestors and itself, one 64-bit word per node.
//
// One warp per sequence.  Node n lives in lane n % 32, slot n / 32 (Q <= 64).  The
// ancestor sets are built by pointer jumping: every node starts with {itself} and a jump
// pointer at its parent; each round ORs in the set of the node it points at and doubles
// the jump, so after 6 rounds every chain of up to 63 steps is covered.  Depth is then the
// population count minus one.  All of it is integer work and bit-exact.
#include "tv_internal.h"

namespace tv {
namespace {

__global__ void __launch_bounds__(128) visibility_kernel(const int32_t* __restrict__ parent,
                                                         int B, int Q,
                                                         uint64_t* __restrict__ anc,
                                                         int32_t* __restrict__ depth,
                                                         uint8_t* __restrict__ mask,
                                                         int32_t* status) {
  const int seq = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (seq >= B) return;  // whole warp leaves together
  const int32_t* par = parent + (int64_t)seq * Q;

  int p[2];
  bool valid = true;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    p[s] = -1;
    if (i < Q) {
      p[s] = par[i];
      valid = valid && (i == 0 ? p[s] == -1 : (p[s] >= 0 && p[s] < i));
    }
  }
  const bool all_ok = __all_sync(0xffffffffu, valid);

  uint64_t A[2];
  int J[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    A[s] = (i < Q) ? (1ull << i) : 0ull;
    J[s] = (i < Q && all_ok) ? p[s] : -1;
  }
#pragma unroll
  for (int round = 0; round < 6; ++round) {
    uint64_t nA[2];
    int nJ[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int src = J[s] < 0 ? lane : J[s];
      const uint64_t a0 = __shfl_sync(0xffffffffu, A[0], src & 31);
      const uint64_t a1 = __shfl_sync(0xffffffffu, A[1], src & 31);
      const int j0 = __shfl_sync(0xffffffffu, J[0], src & 31);
      const int j1 = __shfl_sync(0xffffffffu, J[1], src & 31);
      nA[s] = (src >> 5) ? a1 : a0;
      nJ[s] = (src >> 5) ? j1 : j0;
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (J[s] >= 0) {
        A[s] |= nA[s];
        J[s] = nJ[s];
      }
    }
  }

#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    if (i < Q) {
      anc[(int64_t)seq * Q + i] = all_ok ? A[s] : 0ull;
      depth[(int64_t)seq * Q + i] = all_ok ? (__popcll(A[s]) - 1) : -1;
    }
  }
  if (mask) {
    for (int i = 0; i < Q; ++i) {
      const uint64_t ai0 = __shfl_sync(0xffffffffu, A[0], i & 31);
      const uint64_t ai1 = __shfl_sync(0xffffffffu, A[1], i & 31);
      const uint64_t ai = all_ok ? ((i >> 5) ? ai1 : ai0) : 0ull;
      uint8_t* row = mask + ((int64_t)seq * Q + i) * Q;
      for (int k = lane; k < Q; k += 32) row[k] = (uint8_t)((ai >> k) & 1ull);
    }
  }
  if (!all_ok && lane == 0) report(status, TV_ERR_INVALID_TREE);
}

}  // namespace

cudaError_t launch_visibility(const int32_t* parent, int B, int Q, uint64_t* anc,
                              int32_t* depth, uint8_t* mask, int32_t* status,
                              cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  const int threads = 128;  // 4 sequences per block
  const int blocks = (B * 32 + threads - 1) / threads;
  visibility_kernel<<<blocks, threads, 0, st>>>(parent, B, Q, anc, depth, mask, status);
  return cudaGetLastError();
}

}  // namespace tv
