// fp32 path of the packed LoRA layer: tiled SIMT GEMMs in true fp32 FFMA for fp32 activations and weights.
//
// fp32 inputs with a 1e-4 relative-error budget rule out the tensor cores' tf32 mode
// (its 10-bit mantissa alone gives ~1e-4 per product), so this path computes in true fp32 on the
// FP32 pipes.  Every product is tiled over CTAs of 256 threads: 64 x 64 tiles (4 x 4 outputs per
// thread, K slices of 32), or for a base product large enough for two waves 128 x 128 tiles (8 x 8
// per thread, K slices of 16).  K slices pass through shared memory, the next one fetched into
// registers while the current one is multiplied, and each operand is loaded with the thread mapping
// that makes its contiguous dimension coalesced.  Same definitions as the tensor-core path ("PLoRA: Efficient
// Concurrent LoRA Training for Large Language Models", §2.1, §2.4 and §9.2 Cases 1-4): the base
// products carry the rank term in the same accumulator, job by job over the jobs a row tile
// covers; the per-job products (H, dH, dA, dB) run as one launch over all jobs.
#include "common.cuh"

namespace mlora {

namespace {

constexpr int FTHREADS = 256;

// Output tile T x T per CTA, R x R outputs per thread (16 x 16 threads), K slices of KS.  Small tiles
// for small products and the per-job ones; large tiles (8 x 8 per thread: four FMAs per shared-memory
// load instead of two) for the base products when they make at least two waves of CTAs.
template <int T_, int R_, int KS_>
struct Tile {
  static constexpr int T = T_, R = R_, KS = KS_;
  static constexpr int LD = T + (R == 8 ? 4 : 1);   // padded row: fewer bank conflicts, 16-byte rows for R = 8
  static constexpr int PER = T * KS / FTHREADS;     // elements of each operand slice per thread
  static_assert((T / R) * (T / R) == FTHREADS, "16 x 16 threads per tile");
  // the thread's i-th row (or column) of the tile: four consecutive ones per half tile
  __device__ static __forceinline__ int at(int lane16, int i) { return (i / 4) * (T / 2) + lane16 * 4 + (i % 4); }
};
using Small = Tile<64, 4, 32>;
using Big = Tile<128, 8, 16>;

// A matrix view over rows [r_lo, r_hi) (zero outside): element (i, k) at p[(i - r_lo) * rs + k * cs].
// A second operand is viewed the same way with its output column as i: (k, n) at p[k * rs + (n - r_lo) * cs].
struct View {
  const float* p;
  long long rs, cs;
  long long r_lo, r_hi;
  float scale;
};

// acc += A[m0.., k] * B[k, n0..] over k in [0, K): A is rows x K, B is K x cols (B's rows = k).
// The next K slice is fetched into registers while the current one is multiplied from shared memory.
template <class C>
__device__ __forceinline__ void tile_mac(const View& A, const View& B, long long m0, long long n0, int K,
                                         float (&acc)[C::R][C::R], float (*As)[C::LD], float (*Bs)[C::LD]) {
  constexpr int T = C::T, KS = C::KS, PER = C::PER;
  const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
  const bool a_k = A.cs == 1;   // A contiguous along k
  const bool b_n = B.cs == 1;   // B contiguous along n
  float ra[PER], rb[PER];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = t + u * FTHREADS;
      const int m = a_k ? i / KS : i % T, k = a_k ? i % KS : i / T;
      const long long gm = m0 + m;
      const int gk = k0 + k;
      ra[u] = (gm >= A.r_lo && gm < A.r_hi && gk < K) ? A.scale * A.p[(gm - A.r_lo) * A.rs + gk * A.cs] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = t + u * FTHREADS;
      const int n = b_n ? i % T : i / KS, k = b_n ? i / T : i % KS;
      const long long gn = n0 + n;
      const int gk = k0 + k;
      rb[u] = (gn >= B.r_lo && gn < B.r_hi && gk < K) ? B.p[gk * B.rs + (gn - B.r_lo) * B.cs] : 0.f;
    }
  };
  fetch(0);
  for (int k0 = 0; k0 < K; k0 += KS) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = t + u * FTHREADS;
      As[a_k ? i % KS : i / T][a_k ? i / KS : i % T] = ra[u];
      Bs[b_n ? i / T : i % KS][b_n ? i % T : i / KS] = rb[u];
    }
    __syncthreads();
    if (k0 + KS < K) fetch(k0 + KS);
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      float a[C::R], b[C::R];
      if constexpr (C::R == 8) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float4 av = *reinterpret_cast<const float4*>(&As[k][h * (T / 2) + ty * 4]);
          const float4 bv = *reinterpret_cast<const float4*>(&Bs[k][h * (T / 2) + tx * 4]);
          a[4 * h] = av.x, a[4 * h + 1] = av.y, a[4 * h + 2] = av.z, a[4 * h + 3] = av.w;
          b[4 * h] = bv.x, b[4 * h + 1] = bv.y, b[4 * h + 2] = bv.z, b[4 * h + 3] = bv.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < C::R; ++i) {
          a[i] = As[k][C::at(ty, i)];
          b[i] = Bs[k][C::at(tx, i)];
        }
      }
#pragma unroll
      for (int i = 0; i < C::R; ++i)
#pragma unroll
        for (int j = 0; j < C::R; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
}

// C[m][n] = scale * acc for the thread's outputs inside [0, rows) x [0, cols).
template <class C>
__device__ __forceinline__ void tile_store(float* Cp, long long ldc, long long m0, long long n0, long long rows,
                                           long long cols, float scale, const float (&acc)[C::R][C::R]) {
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int i = 0; i < C::R; ++i) {
    const long long m = m0 + C::at(ty, i);
    if (m >= rows) continue;
#pragma unroll
    for (int j = 0; j < C::R; ++j) {
      const long long n = n0 + C::at(tx, j);
      if (n < cols) Cp[m * ldc + n] = scale * acc[i][j];
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
template <class C>
__global__ void __launch_bounds__(FTHREADS) k_f32_forward(const DevSeg* segs, int n_segs, long long N, int d_in,
                                                          int d_out, const float* X, const float* Wt, const float* H,
                                                          float* Y) {
  __shared__ __align__(16) float As[C::KS][C::LD];
  __shared__ __align__(16) float Bs[C::KS][C::LD];
  const long long m0 = static_cast<long long>(blockIdx.x) * C::T, n0 = static_cast<long long>(blockIdx.y) * C::T;
  float acc[C::R][C::R] = {};
  // X [N, d_in] row-major; W (k, n) = Wt[n][k]
  tile_mac<C>(View{X, d_in, 1, 0, N, 1.f}, View{Wt, 1, d_in, 0, d_out, 1.f}, m0, n0, d_in, acc, As, Bs);
  int j0, j1;
  jobs_of_rows(segs, n_segs, m0, min(N, m0 + C::T), j0, j1);
  for (int j = j0; j <= j1; ++j) {
    const DevSeg sg = segs[j];
    // (s_j H_j)(m, t) for the job's rows only; B_j (t, n) = Bt_j[n][t]
    tile_mac<C>(View{H + sg.h_off, sg.r, 1, sg.off, sg.off + sg.n, sg.s},
             View{sg.Bt, 1, sg.r, 0, d_out, 1.f}, m0, n0, sg.r, acc, As, Bs);
  }
  tile_store<C>(Y, d_out, m0, n0, N, d_out, 1.f, acc);
}

// dX = dY W^T + dH_j A_j^T
template <class C>
__global__ void __launch_bounds__(FTHREADS) k_f32_backward(const DevSeg* segs, int n_segs, long long N, int d_in,
                                                           int d_out, const float* dY, const float* Wt,
                                                           const float* dH, float* dX) {
  __shared__ __align__(16) float As[C::KS][C::LD];
  __shared__ __align__(16) float Bs[C::KS][C::LD];
  const long long m0 = static_cast<long long>(blockIdx.x) * C::T, n0 = static_cast<long long>(blockIdx.y) * C::T;
  float acc[C::R][C::R] = {};
  // dY [N, d_out]; W^T (k = o, n = i) = Wt[o][i]
  tile_mac<C>(View{dY, d_out, 1, 0, N, 1.f}, View{Wt, d_in, 1, 0, d_in, 1.f}, m0, n0, d_out, acc, As, Bs);
  int j0, j1;
  jobs_of_rows(segs, n_segs, m0, min(N, m0 + C::T), j0, j1);
  for (int j = j0; j <= j1; ++j) {
    const DevSeg sg = segs[j];
    // dH_j (m, t); A_j^T (t, i) = At_j[t][i]
    tile_mac<C>(View{dH + sg.h_off, sg.r, 1, sg.off, sg.off + sg.n, 1.f},
             View{sg.At, d_in, 1, 0, d_in, 1.f}, m0, n0, sg.r, acc, As, Bs);
  }
  tile_store<C>(dX, d_in, m0, n0, N, d_in, 1.f, acc);
}

// Per-job products, one CTA per (row tile, column tile, job = blockIdx.z).
//   H_j  [n, r]     = X_j A_j                 (K = d_in)
//   dH_j [n, r]     = s_j dY_j B_j^T          (K = d_out)
//   dBt_j [d_out, r] = s_j dY_j^T H_j          (K = n)
//   dAt_j [r, d_in]  = dH_j^T X_j              (K = n)
__global__ void __launch_bounds__(FTHREADS) k_f32_shrink(const DevSeg* segs, int d_in, const float* X, float* H) {
  using C = Small;
  __shared__ float As[C::KS][C::LD], Bs[C::KS][C::LD];
  const DevSeg sg = segs[blockIdx.z];
  const long long m0 = static_cast<long long>(blockIdx.x) * C::T, n0 = static_cast<long long>(blockIdx.y) * C::T;
  if (m0 >= sg.n || n0 >= sg.r) return;
  float acc[C::R][C::R] = {};
  tile_mac<C>(View{X + sg.off * d_in, d_in, 1, 0, sg.n, 1.f}, View{sg.At, 1, d_in, 0, sg.r, 1.f}, m0, n0, d_in, acc, As,
           Bs);
  tile_store<C>(H + sg.h_off, sg.r, m0, n0, sg.n, sg.r, 1.f, acc);
}

__global__ void __launch_bounds__(FTHREADS) k_f32_dh(const DevSeg* segs, int d_out, const float* dY, float* dH) {
  using C = Small;
  __shared__ float As[C::KS][C::LD], Bs[C::KS][C::LD];
  const DevSeg sg = segs[blockIdx.z];
  const long long m0 = static_cast<long long>(blockIdx.x) * C::T, n0 = static_cast<long long>(blockIdx.y) * C::T;
  if (m0 >= sg.n || n0 >= sg.r) return;
  float acc[C::R][C::R] = {};
  // B_j^T (k = o, n = t) = Bt_j[o][t]
  tile_mac<C>(View{dY + sg.off * d_out, d_out, 1, 0, sg.n, 1.f}, View{sg.Bt, sg.r, 1, 0, sg.r, 1.f}, m0, n0, d_out, acc,
           As, Bs);
  tile_store<C>(dH + sg.h_off, sg.r, m0, n0, sg.n, sg.r, sg.s, acc);
}

__global__ void __launch_bounds__(FTHREADS) k_f32_db(const DevSeg* segs, int d_out, const float* dY, const float* H) {
  using C = Small;
  __shared__ float As[C::KS][C::LD], Bs[C::KS][C::LD];
  const DevSeg sg = segs[blockIdx.z];
  const long long m0 = static_cast<long long>(blockIdx.x) * C::T, n0 = static_cast<long long>(blockIdx.y) * C::T;
  if (n0 >= sg.r) return;
  float acc[C::R][C::R] = {};
  // dY_j^T (o, k = token) = dY[off + k][o];  H_j (k, t)
  tile_mac<C>(View{dY + sg.off * d_out, 1, d_out, 0, d_out, 1.f}, View{H + sg.h_off, sg.r, 1, 0, sg.r, 1.f}, m0, n0, sg.n,
           acc, As, Bs);
  tile_store<C>(sg.dBt, sg.r, m0, n0, d_out, sg.r, sg.s, acc);
}

__global__ void __launch_bounds__(FTHREADS) k_f32_da(const DevSeg* segs, int d_in, const float* X, const float* dH) {
  using C = Small;
  __shared__ float As[C::KS][C::LD], Bs[C::KS][C::LD];
  const DevSeg sg = segs[blockIdx.z];
  const long long m0 = static_cast<long long>(blockIdx.x) * C::T, n0 = static_cast<long long>(blockIdx.y) * C::T;
  if (m0 >= sg.r) return;
  float acc[C::R][C::R] = {};
  // dH_j^T (t, k = token) = dH_j[k][t];  X_j (k, i)
  tile_mac<C>(View{dH + sg.h_off, 1, sg.r, 0, sg.r, 1.f}, View{X + sg.off * d_in, d_in, 1, 0, d_in, 1.f}, m0, n0, sg.n,
           acc, As, Bs);
  tile_store<C>(sg.dAt, d_in, m0, n0, sg.r, d_in, 1.f, acc);
}

template <class C>
unsigned tiles(long long n) { return static_cast<unsigned>((n + C::T - 1) / C::T); }

// large tiles for a base product when they still make at least two waves of CTAs
bool big_tiles(long long rows, long long cols, int num_sms) {
  return static_cast<long long>(tiles<Big>(rows)) * tiles<Big>(cols) >= 2LL * num_sms;
}

}  // namespace

cudaError_t launch_f32_forward(const DevSeg* segs, int n_segs, long long N, int d_in, int d_out, long long h_elems,
                               int max_rank, int max_tokens, int num_sms, const float* X, const float* Wt, float* Y,
                               float* H, cudaStream_t st) {
  if (h_elems > 0)
    k_f32_shrink<<<dim3(tiles<Small>(max_tokens), tiles<Small>(max_rank), n_segs), FTHREADS, 0, st>>>(segs, d_in, X, H);
  if (big_tiles(N, d_out, num_sms))
    k_f32_forward<Big><<<dim3(tiles<Big>(N), tiles<Big>(d_out)), FTHREADS, 0, st>>>(segs, n_segs, N, d_in, d_out, X,
                                                                                     Wt, H, Y);
  else
    k_f32_forward<Small><<<dim3(tiles<Small>(N), tiles<Small>(d_out)), FTHREADS, 0, st>>>(segs, n_segs, N, d_in,
                                                                                         d_out, X, Wt, H, Y);
  return cudaGetLastError();
}

cudaError_t launch_f32_backward(const DevSeg* segs, int n_segs, long long N, int d_in, int d_out, long long h_elems,
                                int max_rank, int max_tokens, int num_sms, const float* X, const float* Wt,
                                const float* dY, const float* H, float* dX, float* dH, cudaStream_t st) {
  if (h_elems > 0)
    k_f32_dh<<<dim3(tiles<Small>(max_tokens), tiles<Small>(max_rank), n_segs), FTHREADS, 0, st>>>(segs, d_out, dY, dH);
  if (big_tiles(N, d_in, num_sms))
    k_f32_backward<Big><<<dim3(tiles<Big>(N), tiles<Big>(d_in)), FTHREADS, 0, st>>>(segs, n_segs, N, d_in, d_out, dY,
                                                                                    Wt, dH, dX);
  else
    k_f32_backward<Small><<<dim3(tiles<Small>(N), tiles<Small>(d_in)), FTHREADS, 0, st>>>(segs, n_segs, N, d_in,
                                                                                        d_out, dY, Wt, dH, dX);
  k_f32_db<<<dim3(tiles<Small>(d_out), tiles<Small>(max_rank), n_segs), FTHREADS, 0, st>>>(segs, d_out, dY, H);
  k_f32_da<<<dim3(tiles<Small>(max_rank), tiles<Small>(d_in), n_segs), FTHREADS, 0, st>>>(segs, d_in, X, dH);
  return cudaGetLastError();
}

}  // namespace mlora
