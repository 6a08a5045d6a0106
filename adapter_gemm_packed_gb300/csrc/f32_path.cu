// fp32 path of the packed LoRA layer: plain FFMA kernels for fp32 activations and weights.
//
// fp32 inputs with a 1e-4 relative-error budget rule out the tensor cores' tf32 mode
// (its 10-bit mantissa alone gives ~1e-4 per product), so this path computes in true fp32.
// It serves small problems, where the layer is latency-bound; every kernel reads the segment
// table directly (no staged images, no bf16 shadows).  Same definitions as the tensor-core
// path ("PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §2.1, §2.4 and
// §9.2 Cases 1-4).
#include "common.cuh"

namespace mlora {

namespace {

// Segment of a token row (segments are sorted and contiguous).
__device__ __forceinline__ int seg_of_row(const DevSeg* segs, int n_segs, long long row) {
  int lo = 0, hi = n_segs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (segs[mid].off <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Job of a packed H element (by h_off).
__device__ __forceinline__ int seg_of_h(const DevSeg* segs, int n_segs, long long e) {
  int lo = 0, hi = n_segs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (segs[mid].h_off <= e) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// H[e] for e in [0, h_elems): one warp per element, reduction over d_in.
__global__ void k_f32_shrink(const DevSeg* segs, int n_segs, long long h_elems, int d_in, const float* X, float* H) {
  const long long e = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (e >= h_elems) return;
  const DevSeg sg = segs[seg_of_h(segs, n_segs, e)];
  const long long local = e - sg.h_off;
  const long long row = sg.off + local / sg.r;
  const int t = static_cast<int>(local % sg.r);
  const float* x = X + row * d_in;
  const float* a = sg.At + static_cast<size_t>(t) * d_in;
  float acc = 0.f;
  for (int k = lane; k < d_in; k += 32) acc = fmaf(x[k], a[k], acc);
  acc = warp_sum(acc);
  if (lane == 0) H[e] = acc;
}

// Y[row][o] = sum_k X[row][k] Wt[o][k] + s_i sum_t H[row][t] Bt_i[o][t]
__global__ void k_f32_forward(const DevSeg* segs, int n_segs, long long N, int d_in, int d_out, const float* X,
                              const float* Wt, const float* H, float* Y) {
  const long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (idx >= N * d_out) return;
  const long long row = idx / d_out;
  const int o = static_cast<int>(idx - row * d_out);
  const DevSeg sg = segs[seg_of_row(segs, n_segs, row)];
  const float* x = X + row * d_in;
  const float* w = Wt + static_cast<size_t>(o) * d_in;
  float acc = 0.f;
  for (int k = 0; k < d_in; ++k) acc = fmaf(x[k], w[k], acc);
  const float* h = H + sg.h_off + (row - sg.off) * sg.r;
  const float* b = sg.Bt + static_cast<size_t>(o) * sg.r;
  float lo = 0.f;
  for (int t = 0; t < sg.r; ++t) lo = fmaf(h[t], b[t], lo);
  Y[idx] = fmaf(sg.s, lo, acc);
}

// dH[e] = s_i sum_o dY[row][o] Bt_i[o][t]: one warp per element.
__global__ void k_f32_dh(const DevSeg* segs, int n_segs, long long h_elems, int d_out, const float* dY, float* dH) {
  const long long e = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (e >= h_elems) return;
  const DevSeg sg = segs[seg_of_h(segs, n_segs, e)];
  const long long local = e - sg.h_off;
  const long long row = sg.off + local / sg.r;
  const int t = static_cast<int>(local % sg.r);
  const float* dy = dY + row * d_out;
  float acc = 0.f;
  for (int o = lane; o < d_out; o += 32) acc = fmaf(dy[o], sg.Bt[static_cast<size_t>(o) * sg.r + t], acc);
  acc = warp_sum(acc);
  if (lane == 0) dH[e] = sg.s * acc;
}

// dX[row][k] = sum_o dY[row][o] Wt[o][k] + sum_t dH[row][t] At_i[t][k]
__global__ void k_f32_backward(const DevSeg* segs, int n_segs, long long N, int d_in, int d_out, const float* dY,
                               const float* Wt, const float* dH, float* dX) {
  const long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (idx >= N * d_in) return;
  const long long row = idx / d_in;
  const int k = static_cast<int>(idx - row * d_in);
  const DevSeg sg = segs[seg_of_row(segs, n_segs, row)];
  const float* dy = dY + row * d_out;
  float acc = 0.f;
  for (int o = 0; o < d_out; ++o) acc = fmaf(dy[o], Wt[static_cast<size_t>(o) * d_in + k], acc);
  const float* dh = dH + sg.h_off + (row - sg.off) * sg.r;
  for (int t = 0; t < sg.r; ++t) acc = fmaf(dh[t], sg.At[static_cast<size_t>(t) * d_in + k], acc);
  dX[idx] = acc;
}

// dBt_i[o][t] = s_i sum_{rows of i} dY[row][o] H[row][t]: one thread per (o, t) of one job (blockIdx.y).
__global__ void k_f32_db(const DevSeg* segs, int d_out, const float* dY, const float* H) {
  const DevSeg sg = segs[blockIdx.y];
  const long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (idx >= static_cast<long long>(d_out) * sg.r) return;
  const int o = static_cast<int>(idx / sg.r);
  const int t = static_cast<int>(idx - static_cast<long long>(o) * sg.r);
  float acc = 0.f;
  for (int n = 0; n < sg.n; ++n)
    acc = fmaf(dY[(sg.off + n) * d_out + o], H[sg.h_off + static_cast<long long>(n) * sg.r + t], acc);
  sg.dBt[idx] = sg.s * acc;
}

// dAt_i[t][k] = sum_{rows of i} dH[row][t] X[row][k]
__global__ void k_f32_da(const DevSeg* segs, int d_in, const float* X, const float* dH) {
  const DevSeg sg = segs[blockIdx.y];
  const long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (idx >= static_cast<long long>(d_in) * sg.r) return;
  const int t = static_cast<int>(idx / d_in);
  const int k = static_cast<int>(idx - static_cast<long long>(t) * d_in);
  float acc = 0.f;
  for (int n = 0; n < sg.n; ++n)
    acc = fmaf(dH[sg.h_off + static_cast<long long>(n) * sg.r + t], X[(sg.off + n) * d_in + k], acc);
  sg.dAt[idx] = acc;
}

inline unsigned blocks(long long threads, int per) { return static_cast<unsigned>((threads + per - 1) / per); }

}  // namespace

cudaError_t launch_f32_forward(const DevSeg* segs, int n_segs, long long N, int d_in, int d_out, long long h_elems,
                               const float* X, const float* Wt, float* Y, float* H, cudaStream_t st) {
  if (h_elems > 0) k_f32_shrink<<<blocks(h_elems * 32, 256), 256, 0, st>>>(segs, n_segs, h_elems, d_in, X, H);
  k_f32_forward<<<blocks(N * d_out, 256), 256, 0, st>>>(segs, n_segs, N, d_in, d_out, X, Wt, H, Y);
  return cudaGetLastError();
}

cudaError_t launch_f32_backward(const DevSeg* segs, int n_segs, long long N, int d_in, int d_out, long long h_elems,
                                int max_rank, const float* X, const float* Wt, const float* dY, const float* H,
                                float* dX, float* dH, cudaStream_t st) {
  if (h_elems > 0) k_f32_dh<<<blocks(h_elems * 32, 256), 256, 0, st>>>(segs, n_segs, h_elems, d_out, dY, dH);
  k_f32_backward<<<blocks(N * d_in, 256), 256, 0, st>>>(segs, n_segs, N, d_in, d_out, dY, Wt, dH, dX);
  dim3 gb(blocks(static_cast<long long>(d_out) * max_rank, 256), n_segs);
  k_f32_db<<<gb, 256, 0, st>>>(segs, d_out, dY, H);
  dim3 ga(blocks(static_cast<long long>(d_in) * max_rank, 256), n_segs);
  k_f32_da<<<ga, 256, 0, st>>>(segs, d_in, X, dH);
  return cudaGetLastError();
}

}  // namespace mlora
