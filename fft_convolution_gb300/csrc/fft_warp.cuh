// fft_warp.cuh -- a 512-point transform held by one warp, its data exchanged
// between stages by register shuffles (__shfl_xor_sync) instead of shared
// memory.
//
// "The Butterfly: One Thread, One Output" (section on the same idea
// elsewhere) notes that the butterfly partners of a pass can be exchanged
// through registers across the lanes of a warp.  Here the 512 points of one
// transform live in one warp, 16 per lane, and the transform is the
// four-step split of "FFT on GPU" (section Fast Fourier Transform) applied
// twice, N = 32 * 16 with the 32-point part split again as 2 * 16:
//   n = n1 + 32 n2 (lane n1, register n2),  k = k2 + 16 c + 256 e,
//   X[k] = sum_a W_2^{a e} W_32^{a c} sum_b W_16^{b c} W_512^{n1 k2}
//          sum_{n2} x[n1 + 32 n2] W_16^{n2 k2},        n1 = a + 2 b.
// 1. the 16-point DFT over n2 in registers, times W_512^{n1 k2};
// 2. four swaps of a lane-index bit with a register-index bit (lane bit
//    1 + i <-> register bit i), each eight complex __shfl_xor_sync, so that
//    register r holds b = r and lane bits 1..4 hold k2;
// 3. the 16-point DFT over b in registers, times W_32^{a c};
// 4. the 2-point DFT over a = lane bit 0 by one __shfl_xor_sync per
//    register.
// Lane (e + 2 k2) then holds X[k2 + 16 c + 256 e] in register c.  No shared
// memory and no block barrier: each warp is independent.
#pragma once

#include "fft_device.cuh"

namespace fftgb {

template <typename V> __device__ __forceinline__ V shfl_xor_c(V v, int mask) {
  V r;
  r.x = __shfl_xor_sync(0xffffffffu, v.x, mask);
  r.y = __shfl_xor_sync(0xffffffffu, v.y, mask);
  return r;
}

// Exchanges register-index bit RB with lane-index bit LB: the value at
// (lane l, register r) moves to the lane whose bit LB is bit RB of r and to
// the register whose bit RB is bit LB of l (other bits unchanged).
template <int RB, int LB, typename V> __device__ __forceinline__ void swap_lane_reg_bit(V *x,
                                                                                     int lane) {
  const bool hi = (lane >> LB) & 1;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    if ((r >> RB) & 1) continue;
    const int r1 = r | (1 << RB);
    const V recv = shfl_xor_c(hi ? x[r] : x[r1], 1 << LB);
    if (hi) x[r] = recv;
    else x[r1] = recv;
  }
}

// On entry x[r] = element lane + 32 r of the input; on exit x[c] = element
// (lane >> 1) + 16 c + 256 (lane & 1) of its DFT (DIR = -1) or of the
// unscaled inverse (DIR = +1).  All 32 lanes of the warp take part.
template <int DIR, typename V> __device__ __forceinline__ void fft512_warp(V *x, int lane) {
  using T = decltype(V::x);
  dft_reg<16, DIR>(x);
  {
    V pw[16];
    powers<16>(twiddle<DIR>((long long)lane, 9, T()), pw);  // W_512^{n1 k2}
#pragma unroll
    for (int k = 1; k < 16; ++k) x[k] = c_mul(x[k], pw[k]);
  }
  swap_lane_reg_bit<0, 1>(x, lane);
  swap_lane_reg_bit<1, 2>(x, lane);
  swap_lane_reg_bit<2, 3>(x, lane);
  swap_lane_reg_bit<3, 4>(x, lane);
  dft_reg<16, DIR>(x);
  const int a = lane & 1;
  {
    V pw[16];
    powers<16>(twiddle<DIR>((long long)a, 5, T()), pw);  // W_32^{a c}
#pragma unroll
    for (int c = 1; c < 16; ++c) x[c] = c_mul(x[c], pw[c]);
  }
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const V p = shfl_xor_c(x[c], 1);
    x[c] = a ? c_sub(p, x[c]) : c_add(x[c], p);
  }
}

}  // namespace fftgb
