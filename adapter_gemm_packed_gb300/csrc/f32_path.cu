// fp32 path of the packed LoRA layer: tiled SIMT GEMMs in true fp32 FFMA for fp32 activations and weights.
//
// fp32 inputs with a 1e-4 relative-error budget rule out the tensor cores' tf32 mode
// (its 10-bit mantissa alone gives ~1e-4 per product), so this path computes in true fp32 on the
// FP32 pipes.  Every product is one 64 x 64 output tile per CTA (256 threads, 4 x 4 outputs each);
// K runs in slices of 32 through shared memory, the next slice fetched into registers while the
// current one is multiplied, and each operand is loaded with the thread mapping that makes its
// contiguous dimension coalesced.  Same definitions as the tensor-core path ("PLoRA: Efficient
// Concurrent LoRA Training for Large Language Models", §2.1, §2.4 and §9.2 Cases 1-4): the base
// products carry the rank term in the same accumulator, job by job over the jobs a row tile
// covers; the per-job products (H, dH, dA, dB) run as one launch over all jobs.
#include "common.cuh"

namespace mlora {

namespace {

constexpr int FT = 64;        // output tile (rows and columns)
constexpr int FK = 32;        // K slice
constexpr int FTHREADS = 256;

// A matrix view over rows [r_lo, r_hi) (zero outside): element (i, k) at p[(i - r_lo) * rs + k * cs].
// A second operand is viewed the same way with its output column as i: (k, n) at p[k * rs + (n - r_lo) * cs].
struct View {
  const float* p;
  long long rs, cs;
  long long r_lo, r_hi;
  float scale;
};

// acc[4][4] += A[m0.., k] * B[k, n0..] over k in [0, K): A is rows x K, B is K x cols (B's rows = k).
// The next K slice is fetched into registers while the current one is multiplied from shared memory.
__device__ __forceinline__ void tile_mac(const View& A, const View& B, long long m0, long long n0, int K,
                                         float (&acc)[4][4], float (*As)[FT + 1], float (*Bs)[FT + 1]) {
  constexpr int PER = FT * FK / FTHREADS;   // elements of each operand slice per thread
  const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
  const bool a_k = A.cs == 1;   // A contiguous along k
  const bool b_n = B.cs == 1;   // B contiguous along n
  float ra[PER], rb[PER];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = t + u * FTHREADS;
      const int m = a_k ? i / FK : i % FT, k = a_k ? i % FK : i / FT;
      const long long gm = m0 + m;
      const int gk = k0 + k;
      ra[u] = (gm >= A.r_lo && gm < A.r_hi && gk < K) ? A.scale * A.p[(gm - A.r_lo) * A.rs + gk * A.cs] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = t + u * FTHREADS;
      const int n = b_n ? i % FT : i / FK, k = b_n ? i / FT : i % FK;
      const long long gn = n0 + n;
      const int gk = k0 + k;
      rb[u] = (gn >= B.r_lo && gn < B.r_hi && gk < K) ? B.p[gk * B.rs + (gn - B.r_lo) * B.cs] : 0.f;
    }
  };
  fetch(0);
  for (int k0 = 0; k0 < K; k0 += FK) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = t + u * FTHREADS;
      As[a_k ? i % FK : i / FT][a_k ? i / FK : i % FT] = ra[u];
      Bs[b_n ? i / FT : i % FK][b_n ? i % FT : i / FK] = rb[u];
    }
    __syncthreads();
    if (k0 + FK < K) fetch(k0 + FK);
#pragma unroll
    for (int k = 0; k < FK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
}

// C[m][n] = scale * acc for the thread's 4 x 4 outputs inside [0, rows) x [0, cols).
__device__ __forceinline__ void tile_store(float* C, long long ldc, long long m0, long long n0, long long rows,
                                           long long cols, float scale, const float (&acc)[4][4]) {
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long m = m0 + ty * 4 + i;
    if (m >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long n = n0 + tx * 4 + j;
      if (n < cols) C[m * ldc + n] = scale * acc[i][j];
    }
  }
}

// Jobs overlapping token rows [lo, hi) (segments are sorted and contiguous).
__device__ __forceinline__ void jobs_of_rows(const DevSeg* segs, int n_segs, long long lo, long long hi, int& j0,
                                             int& j1) {
  int a = 0, b = n_segs - 1;
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (segs[mid].off <= lo) a = mid; else b = mid - 1;
  }
  j0 = a;
  j1 = a;
  while (j1 + 1 < n_segs && segs[j1 + 1].off < hi) ++j1;
}

// Y = X W + s_j H_j B_j, tile (blockIdx.x rows, blockIdx.y columns)
__global__ void __launch_bounds__(FTHREADS) k_f32_forward(const DevSeg* segs, int n_segs, long long N, int d_in,
                                                          int d_out, const float* X, const float* Wt, const float* H,
                                                          float* Y) {
  __shared__ float As[FK][FT + 1], Bs[FK][FT + 1];
  const long long m0 = static_cast<long long>(blockIdx.x) * FT, n0 = static_cast<long long>(blockIdx.y) * FT;
  float acc[4][4] = {};
  // X [N, d_in] row-major; W (k, n) = Wt[n][k]
  tile_mac(View{X, d_in, 1, 0, N, 1.f}, View{Wt, 1, d_in, 0, d_out, 1.f}, m0, n0, d_in, acc, As, Bs);
  int j0, j1;
  jobs_of_rows(segs, n_segs, m0, min(N, m0 + FT), j0, j1);
  for (int j = j0; j <= j1; ++j) {
    const DevSeg sg = segs[j];
    // (s_j H_j)(m, t) for the job's rows only; B_j (t, n) = Bt_j[n][t]
    tile_mac(View{H + sg.h_off, sg.r, 1, sg.off, sg.off + sg.n, sg.s},
             View{sg.Bt, 1, sg.r, 0, d_out, 1.f}, m0, n0, sg.r, acc, As, Bs);
  }
  tile_store(Y, d_out, m0, n0, N, d_out, 1.f, acc);
}

// dX = dY W^T + dH_j A_j^T
__global__ void __launch_bounds__(FTHREADS) k_f32_backward(const DevSeg* segs, int n_segs, long long N, int d_in,
                                                           int d_out, const float* dY, const float* Wt,
                                                           const float* dH, float* dX) {
  __shared__ float As[FK][FT + 1], Bs[FK][FT + 1];
  const long long m0 = static_cast<long long>(blockIdx.x) * FT, n0 = static_cast<long long>(blockIdx.y) * FT;
  float acc[4][4] = {};
  // dY [N, d_out]; W^T (k = o, n = i) = Wt[o][i]
  tile_mac(View{dY, d_out, 1, 0, N, 1.f}, View{Wt, d_in, 1, 0, d_in, 1.f}, m0, n0, d_out, acc, As, Bs);
  int j0, j1;
  jobs_of_rows(segs, n_segs, m0, min(N, m0 + FT), j0, j1);
  for (int j = j0; j <= j1; ++j) {
    const DevSeg sg = segs[j];
    // dH_j (m, t); A_j^T (t, i) = At_j[t][i]
    tile_mac(View{dH + sg.h_off, sg.r, 1, sg.off, sg.off + sg.n, 1.f},
             View{sg.At, d_in, 1, 0, d_in, 1.f}, m0, n0, sg.r, acc, As, Bs);
  }
  tile_store(dX, d_in, m0, n0, N, d_in, 1.f, acc);
}

// Per-job products, one CTA per (row tile, column tile, job = blockIdx.z).
//   H_j  [n, r]     = X_j A_j                 (K = d_in)
//   dH_j [n, r]     = s_j dY_j B_j^T          (K = d_out)
//   dBt_j [d_out, r] = s_j dY_j^T H_j          (K = n)
//   dAt_j [r, d_in]  = dH_j^T X_j              (K = n)
__global__ void __launch_bounds__(FTHREADS) k_f32_shrink(const DevSeg* segs, int d_in, const float* X, float* H) {
  __shared__ float As[FK][FT + 1], Bs[FK][FT + 1];
  const DevSeg sg = segs[blockIdx.z];
  const long long m0 = static_cast<long long>(blockIdx.x) * FT, n0 = static_cast<long long>(blockIdx.y) * FT;
  if (m0 >= sg.n || n0 >= sg.r) return;
  float acc[4][4] = {};
  tile_mac(View{X + sg.off * d_in, d_in, 1, 0, sg.n, 1.f}, View{sg.At, 1, d_in, 0, sg.r, 1.f}, m0, n0, d_in, acc, As,
           Bs);
  tile_store(H + sg.h_off, sg.r, m0, n0, sg.n, sg.r, 1.f, acc);
}

__global__ void __launch_bounds__(FTHREADS) k_f32_dh(const DevSeg* segs, int d_out, const float* dY, float* dH) {
  __shared__ float As[FK][FT + 1], Bs[FK][FT + 1];
  const DevSeg sg = segs[blockIdx.z];
  const long long m0 = static_cast<long long>(blockIdx.x) * FT, n0 = static_cast<long long>(blockIdx.y) * FT;
  if (m0 >= sg.n || n0 >= sg.r) return;
  float acc[4][4] = {};
  // B_j^T (k = o, n = t) = Bt_j[o][t]
  tile_mac(View{dY + sg.off * d_out, d_out, 1, 0, sg.n, 1.f}, View{sg.Bt, sg.r, 1, 0, sg.r, 1.f}, m0, n0, d_out, acc,
           As, Bs);
  tile_store(dH + sg.h_off, sg.r, m0, n0, sg.n, sg.r, sg.s, acc);
}

__global__ void __launch_bounds__(FTHREADS) k_f32_db(const DevSeg* segs, int d_out, const float* dY, const float* H) {
  __shared__ float As[FK][FT + 1], Bs[FK][FT + 1];
  const DevSeg sg = segs[blockIdx.z];
  const long long m0 = static_cast<long long>(blockIdx.x) * FT, n0 = static_cast<long long>(blockIdx.y) * FT;
  if (n0 >= sg.r) return;
  float acc[4][4] = {};
  // dY_j^T (o, k = token) = dY[off + k][o];  H_j (k, t)
  tile_mac(View{dY + sg.off * d_out, 1, d_out, 0, d_out, 1.f}, View{H + sg.h_off, sg.r, 1, 0, sg.r, 1.f}, m0, n0, sg.n,
           acc, As, Bs);
  tile_store(sg.dBt, sg.r, m0, n0, d_out, sg.r, sg.s, acc);
}

__global__ void __launch_bounds__(FTHREADS) k_f32_da(const DevSeg* segs, int d_in, const float* X, const float* dH) {
  __shared__ float As[FK][FT + 1], Bs[FK][FT + 1];
  const DevSeg sg = segs[blockIdx.z];
  const long long m0 = static_cast<long long>(blockIdx.x) * FT, n0 = static_cast<long long>(blockIdx.y) * FT;
  if (m0 >= sg.r) return;
  float acc[4][4] = {};
  // dH_j^T (t, k = token) = dH_j[k][t];  X_j (k, i)
  tile_mac(View{dH + sg.h_off, 1, sg.r, 0, sg.r, 1.f}, View{X + sg.off * d_in, d_in, 1, 0, d_in, 1.f}, m0, n0, sg.n,
           acc, As, Bs);
  tile_store(sg.dAt, d_in, m0, n0, sg.r, d_in, 1.f, acc);
}

inline unsigned tiles(long long n) { return static_cast<unsigned>((n + FT - 1) / FT); }

}  // namespace

cudaError_t launch_f32_forward(const DevSeg* segs, int n_segs, long long N, int d_in, int d_out, long long h_elems,
                               int max_rank, int max_tokens, const float* X, const float* Wt, float* Y, float* H,
                               cudaStream_t st) {
  if (h_elems > 0)
    k_f32_shrink<<<dim3(tiles(max_tokens), tiles(max_rank), n_segs), FTHREADS, 0, st>>>(segs, d_in, X, H);
  k_f32_forward<<<dim3(tiles(N), tiles(d_out)), FTHREADS, 0, st>>>(segs, n_segs, N, d_in, d_out, X, Wt, H, Y);
  return cudaGetLastError();
}

cudaError_t launch_f32_backward(const DevSeg* segs, int n_segs, long long N, int d_in, int d_out, long long h_elems,
                                int max_rank, int max_tokens, const float* X, const float* Wt, const float* dY,
                                const float* H, float* dX, float* dH, cudaStream_t st) {
  if (h_elems > 0)
    k_f32_dh<<<dim3(tiles(max_tokens), tiles(max_rank), n_segs), FTHREADS, 0, st>>>(segs, d_out, dY, dH);
  k_f32_backward<<<dim3(tiles(N), tiles(d_in)), FTHREADS, 0, st>>>(segs, n_segs, N, d_in, d_out, dY, Wt, dH, dX);
  k_f32_db<<<dim3(tiles(d_out), tiles(max_rank), n_segs), FTHREADS, 0, st>>>(segs, d_out, dY, H);
  k_f32_da<<<dim3(tiles(max_rank), tiles(d_in), n_segs), FTHREADS, 0, st>>>(segs, d_in, X, dH);
  return cudaGetLastError();
}

}  // namespace mlora
