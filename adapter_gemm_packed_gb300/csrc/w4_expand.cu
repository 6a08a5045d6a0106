// Expansion of a 4-bit base weight to bf16 W^T once per call (the default for 4-bit-base
// plans): Wt [d_out, d_in] bf16 = bf16(q[o][k] * Wscale[k / 64][o]), the layout the bf16 base
// GEMMs read, so that the rest of the layer is the bf16 path unchanged.
//
// Pure streaming: 0.5 B of codes + 4/64 B of scales read and 2 B written per weight.  A block
// of 128 threads covers 512 code words (4096 weights) of one output row; thread t takes words
// t, t + 128, t + 256, t + 384, so each warp instruction reads 128 contiguous bytes of codes and
// writes 512 contiguous bytes of W^T, and all four loads are in flight before any arithmetic.
// The scales of one row are d_out floats apart; neighbouring rows' blocks share their sectors
// through L2.
#include "common.cuh"
#include "w4.cuh"

namespace mlora {

namespace {

constexpr int EXP_THREADS = 128;
constexpr int EXP_WORDS = 4;   // code words (8 weights each) per thread

__global__ void __launch_bounds__(EXP_THREADS) k_w4_expand(const uint32_t* __restrict__ Wq, const float* __restrict__ Ws,
                                                           uint4* __restrict__ Wt, int d_in, int d_out) {
  // the output may still be read by the previous call's GEMM: wait for it before writing
  griddep_wait();
  griddep_launch_dependents();
  const uint64_t magic2 = w4::magic_pair();
  const int wpr = d_in / 8;   // code words per output row
  const int kw0 = blockIdx.x * (EXP_THREADS * EXP_WORDS) + threadIdx.x;
  for (int o = blockIdx.y; o < d_out; o += gridDim.y) {
    const long long row = static_cast<long long>(o) * wpr;
    uint32_t w[EXP_WORDS];
    float sc[EXP_WORDS];
#pragma unroll
    for (int j = 0; j < EXP_WORDS; ++j) {
      const int kw = kw0 + j * EXP_THREADS;
      if (kw < wpr) {
        w[j] = __ldcs(Wq + row + kw);
        sc[j] = __ldg(Ws + static_cast<long long>(kw >> 3) * d_out + o);
      }
    }
#pragma unroll
    for (int j = 0; j < EXP_WORDS; ++j) {
      const int kw = kw0 + j * EXP_THREADS;
      if (kw < wpr) Wt[row + kw] = w4::expand8(w[j], sc[j], magic2);
    }
  }
}

}  // namespace

cudaError_t launch_w4_expand(const void* Wq, const float* Ws, __nv_bfloat16* Wt, int d_in, int d_out, int num_sms,
                             cudaStream_t st, bool pdl) {
  (void)num_sms;
  const int wpr = d_in / 8;
  const unsigned gx = static_cast<unsigned>((wpr + EXP_THREADS * EXP_WORDS - 1) / (EXP_THREADS * EXP_WORDS));
  const unsigned gy = static_cast<unsigned>(d_out < 65535 ? d_out : 65535);
  return launch_k(k_w4_expand, dim3(gx, gy), dim3(EXP_THREADS), 0, st, pdl, static_cast<const uint32_t*>(Wq), Ws,
                  reinterpret_cast<uint4*>(Wt), d_in, d_out);
}

}  // namespace mlora
