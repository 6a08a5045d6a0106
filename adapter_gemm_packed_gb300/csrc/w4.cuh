// Expansion of the 4-bit base's codes to bf16, shared by the expansion kernel (w4_expand.cu)
// and the converter warps of the fused CTA-pair GEMMs (gemm_2sm_w4.cu).
//
// Format (the reading this library takes of the 4-bit / QLoRA base of "PLoRA: Efficient
// Concurrent LoRA Training for Large Language Models", §5 and §11.3, which do not fix one):
// signed codes q in [-8, 7], two's complement, two per byte with the even k in the low nibble,
// one fp32 scale per 64 consecutive d_in entries of each output column, and
// W[k][o] = bf16(q * scale) with the product rounded to fp32 and then to nearest bf16.
#pragma once
#include <cstdint>

namespace mlora {
namespace w4 {

// Two codes at the same byte position B of `lo` / `hi` (each byte holds code + 8, 0..15) as a
// bf16 pair (lo's in the low half): the byte is placed in the low mantissa bits of the float
// 2^23 + byte, and subtracting 2^23 + 8 leaves the signed code exactly; one fp32 multiply by the
// scale (packed twice in s2) and one round to bf16 follow.
template <int B>
__device__ __forceinline__ uint32_t pair_bf16(uint32_t lo, uint32_t hi, uint64_t magic2, uint64_t s2) {
  uint32_t r;
  asm("{\n\t.reg .b32 x0, x1;\n\t.reg .b64 v;\n\t"
      "prmt.b32 x0, %1, 0x4B000000, %3;\n\t"
      "prmt.b32 x1, %2, 0x4B000000, %3;\n\t"
      "mov.b64 v, {x0, x1};\n\t"
      "sub.rn.f32x2 v, v, %4;\n\t"
      "mul.rn.f32x2 v, v, %5;\n\t"
      "mov.b64 {x0, x1}, v;\n\t"
      "cvt.rn.bf16x2.f32 %0, x1, x0;\n\t}"
      : "=r"(r)
      : "r"(lo), "r"(hi), "n"(0x7540 + B), "l"(magic2), "l"(s2));
  return r;
}

// (2^23 + 8, 2^23 + 8) as a packed pair, the offset pair_bf16 subtracts.
__device__ __forceinline__ uint64_t magic_pair() {
  uint64_t m;
  asm("mov.b64 %0, {%1, %1};" : "=l"(m) : "f"(8388616.0f));
  return m;
}

// The eight codes of one 32-bit word (code e in nibble e) times s, as eight bf16 in code order.
__device__ __forceinline__ uint4 expand8(uint32_t w, float s, uint64_t magic2) {
  const uint32_t ev = (w & 0x0F0F0F0Fu) ^ 0x08080808u;          // codes 0, 2, 4, 6, each + 8
  const uint32_t od = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;   // codes 1, 3, 5, 7, each + 8
  uint64_t s2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(s));
  return make_uint4(pair_bf16<0>(ev, od, magic2, s2), pair_bf16<1>(ev, od, magic2, s2),
                    pair_bf16<2>(ev, od, magic2, s2), pair_bf16<3>(ev, od, magic2, s2));
}

}  // namespace w4
}  // namespace mlora
