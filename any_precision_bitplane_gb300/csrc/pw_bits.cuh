// Bit-matrix helpers shared by the decode and prefill kernels: q stacked
// bitplane words (32 columns of one row) -> one q-bit index per byte.
#pragma once

#include <cstdint>

namespace pw {

// Byte transpose of four 32-bit words: out[b] = {a0.byte b, a1.byte b,
// a2.byte b, a3.byte b}.
__device__ __forceinline__ void byte_transpose4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t (&out)[4]) {
  const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);
  const uint32_t t2 = __byte_perm(a2, a3, 0x5140), t3 = __byte_perm(a2, a3, 0x7362);
  out[0] = __byte_perm(t0, t2, 0x5410);
  out[1] = __byte_perm(t0, t2, 0x7632);
  out[2] = __byte_perm(t1, t3, 0x5410);
  out[3] = __byte_perm(t1, t3, 0x7632);
}

// Multipliers for the bit transpose, passed as kernel parameters so that
// the compiler keeps them as integer multiplies: x >> s == umulhi(x, 2^(32-s))
// and x << s == x * 2^s, which run on the multiply-add pipe and leave the
// logic pipe to the XOR / AND / byte-permute work.
struct BitConsts {
  uint32_t hi7, mul7;     // 2^25, 2^7 + 1
  uint32_t hi14, mul14;   // 2^18, 2^14 + 1
  uint32_t hi4, mul4;     // 2^28, 2^4
  uint32_t shl[3];        // 2^1, 2^2, 2^4:          x << d  == x * shl
  uint32_t shr[3];        // 2^31, 2^30, 2^28:       x >> d  == umulhi(x, shr)
};

inline BitConsts make_bit_consts() {
  BitConsts bc;
  bc.hi7 = 1u << 25;
  bc.mul7 = (1u << 7) + 1u;
  bc.hi14 = 1u << 18;
  bc.mul14 = (1u << 14) + 1u;
  bc.hi4 = 1u << 28;
  bc.mul4 = 1u << 4;
  for (int i = 0; i < 3; ++i) {
    bc.shl[i] = 1u << (1 << i);
    bc.shr[i] = 1u << (32 - (1 << i));
  }
  return bc;
}

// ---- register-index / bit-position transpose ---------------------------------
//
// View R[0..n) as a matrix with one bit per (register r, bit position t).
// swap_stage<I> exchanges bit I of the register index with bit I of the bit
// position: for the register pair lo = R[r] (bit I of r clear) and
// hi = R[r + 2^I], lo's bits at positions with bit I set trade places with
// hi's bits at the positions 2^I lower.  Two shifts (integer multiplies by
// kernel-parameter constants, so they run on the multiply-add pipe) and two
// bit selects.  When one register is the constant 0 the compiler folds the
// stage to three operations, or to nothing when both are.
template <int I>
__device__ __forceinline__ void swap_stage(uint32_t& lo, uint32_t& hi, const BitConsts& bc) {
  constexpr uint32_t M = I == 0 ? 0x55555555u : I == 1 ? 0x33333333u : 0x0F0F0F0Fu;
  const uint32_t hs = hi * bc.shl[I];
  const uint32_t ls = __umulhi(lo, bc.shr[I]);
  lo = (lo & M) | (hs & ~M);
  hi = (ls & M) | (hi & ~M);
}

// Q <= 4 plane words of one row (P[0] = most significant plane) covering the
// 32 columns of a word -> 4-bit indices: nibble n of N[r] is the Q-bit index
// of column 4n + r (bit 3 is 0 when Q < 4).  Register r starts as plane
// Q-1-r, the plane feeding index bit r; swapping register-index bits 0 and 1
// with position bits 0 and 1 moves every column's Q bits into one nibble.
template <int Q>
__device__ __forceinline__ void planes_to_nibbles(const uint32_t (&P)[Q], uint32_t (&N)[4],
                                                  const BitConsts& bc) {
  static_assert(Q >= 1 && Q <= 4, "nibble indices hold at most 4 bits");
#pragma unroll
  for (int r = 0; r < 4; ++r) N[r] = (r < Q) ? P[Q - 1 - r] : 0u;
  swap_stage<0>(N[0], N[1], bc);
  swap_stage<0>(N[2], N[3], bc);
  swap_stage<1>(N[0], N[2], bc);
  swap_stage<1>(N[1], N[3], bc);
}

// Q <= 8 plane words of one row -> 8-bit indices: byte b of B[r] is the
// Q-bit index of column 8b + r.  Same construction with register-index bits
// 0, 1 and 2 swapped with position bits 0, 1 and 2.
template <int Q>
__device__ __forceinline__ void planes_to_bytes(const uint32_t (&P)[Q], uint32_t (&B)[8],
                                                const BitConsts& bc) {
  static_assert(Q >= 1 && Q <= 8, "at most 8 planes");
#pragma unroll
  for (int r = 0; r < 8; ++r) B[r] = (r < Q) ? P[Q - 1 - r] : 0u;
#pragma unroll
  for (int r = 0; r < 8; r += 2) swap_stage<0>(B[r], B[r + 1], bc);
  swap_stage<1>(B[0], B[2], bc);
  swap_stage<1>(B[1], B[3], bc);
  swap_stage<1>(B[4], B[6], bc);
  swap_stage<1>(B[5], B[7], bc);
#pragma unroll
  for (int r = 0; r < 4; ++r) swap_stage<2>(B[r], B[r + 4], bc);
}

// Column order the two index forms produce, as positions within a word
// column of 32.  The kernels lay their activations out in these orders, so
// each product pairs a weight with its own column:
//   byte form:   the weight in byte b of B[r] (column 8b + r) sits at
//                position 4r + b (B[r] pairs with the 4 activations at 4r);
//   nibble form: byte j of N[r] pairs columns 8j + r (low nibble) and
//                8j + 4 + r (high nibble); they sit at positions 8r + 2j and
//                8r + 2j + 1.
__host__ __device__ __forceinline__ int byte_form_position(int col) {
  return 4 * (col & 7) + (col >> 3);
}
__host__ __device__ __forceinline__ int nibble_form_position(int col) {
  return 8 * (col & 3) + 2 * (col >> 3) + ((col >> 2) & 1);
}

// Transpose of the 8x8 bit matrix held in (lo, hi): byte r = matrix row r,
// bit c = column c  ->  byte c = column c, bit r = row r.  Two delta-swap
// stages inside each half and one nibble exchange between the halves.  In a
// delta swap the swapped bits t and t << s never overlap, so
// x ^ t ^ (t << s) is x ^ (t * (2^s + 1)).
__device__ __forceinline__ void delta_swap(uint32_t& x, uint32_t hi_mul, uint32_t mul, uint32_t m) {
  const uint32_t t = (x ^ __umulhi(x, hi_mul)) & m;
  x ^= t * mul;
}

__device__ __forceinline__ void bit_transpose8(uint32_t& lo, uint32_t& hi, const BitConsts& bc) {
  delta_swap(lo, bc.hi7, bc.mul7, 0x00AA00AAu);
  delta_swap(hi, bc.hi7, bc.mul7, 0x00AA00AAu);
  delta_swap(lo, bc.hi14, bc.mul14, 0x0000CCCCu);
  delta_swap(hi, bc.hi14, bc.mul14, 0x0000CCCCu);
  const uint32_t l = lo;
  lo = (lo & 0x0F0F0F0Fu) | ((hi * bc.mul4) & 0xF0F0F0F0u);
  hi = (hi & 0xF0F0F0F0u) | (__umulhi(l, bc.hi4) & 0x0F0F0F0Fu);
}

// Q plane words of one row (P[0] = most significant plane) covering 32
// columns -> the q-bit index of every column, one per byte: byte j of ib[m]
// is the index of column 4m + j.  Plane p feeds bit (Q-1-p) of the index;
// for Q <= 4 half of the matrix is zero and the compiler folds it away.
template <int Q>
__device__ __forceinline__ void planes_to_index_bytes(const uint32_t (&P)[Q], uint32_t (&ib)[8],
                                                      const BitConsts& bc) {
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = (i < Q) ? P[Q - 1 - i] : 0u;
  uint32_t A[4], B[4];
  byte_transpose4(r[0], r[1], r[2], r[3], A);
  byte_transpose4(r[4], r[5], r[6], r[7], B);
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    uint32_t lo = A[b], hi = B[b];
    bit_transpose8(lo, hi, bc);
    ib[2 * b] = lo;
    ib[2 * b + 1] = hi;
  }
}

}  // namespace pw
