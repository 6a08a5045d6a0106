// Expansion of a 4-bit base weight to bf16 W^T once per call (the default for 4-bit-base
// plans): Wt [d_out, d_in] bf16 = bf16(q[o][k] * Wscale[k / 64][o]), the layout the bf16 base
// GEMMs read, so that the rest of the layer is the bf16 path unchanged.
//
// Pure streaming: 0.5 B of codes + 4/64 B of scales read and 2 B written per weight; one
// thread per 16 bytes of codes (32 weights of one output row, 64 bytes of output), so a warp
// reads 512 contiguous bytes of codes and writes 2 KB contiguous.  The scales of one row are
// d_out floats apart; neighbouring rows' warps share their sectors through L2.
#include "common.cuh"
#include "w4.cuh"

namespace mlora {

namespace {

__global__ void __launch_bounds__(256) k_w4_expand(const uint4* __restrict__ Wq, const float* __restrict__ Ws,
                                                   uint4* __restrict__ Wt, int d_in, int d_out) {
  // the output may still be read by the previous call's GEMM: wait for it before writing
  griddep_wait();
  griddep_launch_dependents();
  const uint64_t magic2 = w4::magic_pair();
  const int upr = d_in / 32;   // 16-byte code units per output row
  const long long total = static_cast<long long>(d_out) * upr;
  for (long long u = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; u < total;
       u += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int o = static_cast<int>(u / upr), c = static_cast<int>(u % upr);
    const uint4 w = __ldcs(Wq + u);
    const float s = __ldg(Ws + static_cast<long long>(c >> 1) * d_out + o);
    uint4* dst = Wt + 4 * u;
    dst[0] = w4::expand8(w.x, s, magic2);
    dst[1] = w4::expand8(w.y, s, magic2);
    dst[2] = w4::expand8(w.z, s, magic2);
    dst[3] = w4::expand8(w.w, s, magic2);
  }
}

}  // namespace

cudaError_t launch_w4_expand(const void* Wq, const float* Ws, __nv_bfloat16* Wt, int d_in, int d_out, int num_sms,
                             cudaStream_t st, bool pdl) {
  const long long units = static_cast<long long>(d_out) * (d_in / 32);
  long long grid = (units + 255) / 256;
  if (grid > static_cast<long long>(num_sms) * 8) grid = static_cast<long long>(num_sms) * 8;
  if (grid < 1) grid = 1;
  return launch_k(k_w4_expand, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, pdl,
                  static_cast<const uint4*>(Wq), Ws, reinterpret_cast<uint4*>(Wt), d_in, d_out);
}

}  // namespace mlora
