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
};

inline BitConsts make_bit_consts() {
  BitConsts bc;
  bc.hi7 = 1u << 25;
  bc.mul7 = (1u << 7) + 1u;
  bc.hi14 = 1u << 18;
  bc.mul14 = (1u << 14) + 1u;
  bc.hi4 = 1u << 28;
  bc.mul4 = 1u << 4;
  return bc;
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
