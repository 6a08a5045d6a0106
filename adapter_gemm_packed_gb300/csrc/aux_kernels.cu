// Memory-bound helper kernels of the packed LoRA layer:
//  * bf16 shadows of the fp32 adapter masters in the packed rank space (the operands the
//    tensor-core engine reads through TMA; the backward reads them MN-major);
//  * rebuild of the staged Htilde images from the saved activation H (backward);
//  * the per-adapter AdamW step over every A_i and B_i ("PLoRA: Efficient Concurrent LoRA
//    Training for Large Language Models", §8: moment, velocity and gradient per parameter;
//    the step order is PyTorch's decoupled-weight-decay AdamW).
#include "common.cuh"

namespace mlora {

namespace {

// At_all [C_total, d_in] bf16: row c = At[c - c0] of the adapter owning packed column c, zero in
// padding.
__global__ void k_pack_at(const DevSub* __restrict__ subs, const int* __restrict__ col_sub, int C_total, int d_in,
                          __nv_bfloat16* __restrict__ at_all) {
  griddep_wait();
  griddep_launch_dependents();
  const int d8 = d_in / 8;
  const long long total = static_cast<long long>(C_total) * d8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i / d8);
    const int k = static_cast<int>(i - static_cast<long long>(c) * d8) * 8;
    const int a = col_sub[c];
    uint4 o = make_uint4(0, 0, 0, 0);
    if (a >= 0) {
      const DevSub& sb = subs[a];
      const float4* src = reinterpret_cast<const float4*>(sb.At + static_cast<size_t>(c - sb.c0) * d_in + k);
      const float4 x = src[0], y = src[1];
      o.x = pack_bf16x2(x.x, x.y);
      o.y = pack_bf16x2(x.z, x.w);
      o.z = pack_bf16x2(y.x, y.y);
      o.w = pack_bf16x2(y.z, y.w);
    }
    *reinterpret_cast<uint4*>(at_all + static_cast<size_t>(c) * d_in + k) = o;
  }
}

// Bt_all [d_out, C_total] bf16: Bt_all[o][c] = Bt[o - o_lo][c - c0] of the adapter owning packed
// column c when output column o lies in that adapter's range [o_lo, o_hi), else zero (padding,
// and the other projections' columns of a shared-input pack).
__global__ void k_pack_bt(const DevSub* __restrict__ subs, const int* __restrict__ col_sub, int C_total, int d_out,
                          __nv_bfloat16* __restrict__ bt_all) {
  griddep_wait();
  griddep_launch_dependents();
  const int c8 = C_total / 8;
  const long long total = static_cast<long long>(d_out) * c8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int o = static_cast<int>(i / c8);
    const int c = static_cast<int>(i - static_cast<long long>(o) * c8) * 8;
    float f[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int a = col_sub[c + u];
      f[u] = 0.f;
      if (a >= 0) {
        const DevSub& sb = subs[a];
        if (o >= sb.o_lo && o < sb.o_hi) f[u] = sb.Bt[static_cast<size_t>(o - sb.o_lo) * sb.r + (c + u - sb.c0)];
      }
    }
    uint4 v;
    v.x = pack_bf16x2(f[0], f[1]);
    v.y = pack_bf16x2(f[2], f[3]);
    v.z = pack_bf16x2(f[4], f[5]);
    v.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4*>(bt_all + static_cast<size_t>(o) * C_total + c) = v;
  }
}

// Staged Htilde images from H (row-major [128 x 64] bf16 blocks):
// image (tile t, chunk q) row r col u = s_c H_j[row - off_j][c - c_j], c = 64q + u, s_c the scale of
// the adapter owning column c, when token row (128 t + r) belongs to job j and column c lies in
// job j's rank window, else 0.
__global__ void k_h_images(const DevSeg* __restrict__ segs, const float* __restrict__ col_scale,
                           const MTile* __restrict__ mtiles, const int* __restrict__ img_tile, long long N,
                           const float* __restrict__ H, uint8_t* __restrict__ img_out) {
  griddep_wait();
  griddep_launch_dependents();
  const int img = blockIdx.x;
  const int t = img_tile[img];
  const MTile mt = mtiles[t];
  const int q = mt.q_lo + (img - mt.img_off);
  const int rit = threadIdx.x;   // 128 threads: one row each
  const long long row = static_cast<long long>(t) * BM + rit;
  int c_lo = 0, c_hi = 0;
  const float* hrow = nullptr;
  if (row < N) {
    int j = mt.seg_first;
    while (j < mt.seg_last && row >= segs[j + 1].off) ++j;
    const DevSeg& sg = segs[j];
    c_lo = sg.c;
    c_hi = sg.c + sg.r;
    hrow = H + sg.h_off + (row - sg.off) * sg.r - sg.c;
  }
  uint8_t* base = img_out + static_cast<size_t>(img) * IMG_BYTES;
#pragma unroll
  for (int k8 = 0; k8 < 8; ++k8) {
    uint32_t pk[4];
#pragma unroll
    for (int u = 0; u < 8; u += 2) {
      const int c0 = q * CHUNK_COLS + k8 * 8 + u, c1 = c0 + 1;
      const float a0 = (c0 >= c_lo && c0 < c_hi) ? col_scale[c0] * hrow[c0] : 0.f;
      const float a1 = (c1 >= c_lo && c1 < c_hi) ? col_scale[c1] * hrow[c1] : 0.f;
      pk[u / 2] = pack_bf16x2(a0, a1);
    }
    *reinterpret_cast<uint4*>(base + rit * (CHUNK_COLS * 2) + k8 * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

// AdamW over a list of <= ADAM_CHUNK-element pieces of every adapter's A and B.
__global__ void k_adamw(const AdamItem* __restrict__ items, int n_items, float lr, float beta1, float beta2,
                        float eps, float decay, float bc1, float bc2, __nv_bfloat16* __restrict__ at_all,
                        __nv_bfloat16* __restrict__ bt_all, int C_total) {
  griddep_wait();
  griddep_launch_dependents();
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const AdamItem w = items[it];
    // with shadows to refresh, each new value also goes to its bf16 copy in the packed rank space
    // (rounded as the pack kernels round, so a later forward sees what a fresh pack would give)
    const int kind = at_all ? w.sh_kind : 0;
    const int n4 = w.count >> 2;
    float4* p4 = reinterpret_cast<float4*>(w.p);
    const float4* g4 = reinterpret_cast<const float4*>(w.g);
    float4* m4 = reinterpret_cast<float4*>(w.m);
    float4* v4 = reinterpret_cast<float4*>(w.v);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      float4 p = p4[i];
      const float4 g = g4[i];
      float4 m = m4[i], v = v4[i];
      float* pp = &p.x;
      const float* gg = &g.x;
      float* mm = &m.x;
      float* vv = &v.x;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float gu = gg[u];
        const float pd = pp[u] * decay;
        const float mu = beta1 * mm[u] + (1.f - beta1) * gu;
        const float vu = beta2 * vv[u] + (1.f - beta2) * gu * gu;
        const float mhat = mu / bc1;
        const float vhat = vu / bc2;
        pp[u] = pd - lr * mhat / (sqrtf(vhat) + eps);
        mm[u] = mu;
        vv[u] = vu;
      }
      p4[i] = p;
      m4[i] = m;
      v4[i] = v;
      if (kind == 1) {
        *reinterpret_cast<uint2*>(at_all + w.sh_base + 4 * i) = make_uint2(pack_bf16x2(p.x, p.y), pack_bf16x2(p.z, p.w));
      } else if (kind == 2) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = w.sh_e0 + 4 * i + u;
          const int o = e / w.sh_r;
          bt_all[w.sh_base + static_cast<long long>(o) * C_total + (e - o * w.sh_r)] = __float2bfloat16_rn(pp[u]);
        }
      }
    }
    for (int i = (n4 << 2) + threadIdx.x; i < w.count; i += blockDim.x) {
      const float gu = w.g[i];
      const float pd = w.p[i] * decay;
      const float mu = beta1 * w.m[i] + (1.f - beta1) * gu;
      const float vu = beta2 * w.v[i] + (1.f - beta2) * gu * gu;
      const float pn = pd - lr * (mu / bc1) / (sqrtf(vu / bc2) + eps);
      w.p[i] = pn;
      w.m[i] = mu;
      w.v[i] = vu;
      if (kind == 1) {
        at_all[w.sh_base + i] = __float2bfloat16_rn(pn);
      } else if (kind == 2) {
        const int e = w.sh_e0 + i;
        const int o = e / w.sh_r;
        bt_all[w.sh_base + static_cast<long long>(o) * C_total + (e - o * w.sh_r)] = __float2bfloat16_rn(pn);
      }
    }
  }
}

inline int grid_for(long long work, int threads, int num_sms) {
  long long b = (work + threads - 1) / threads;
  long long cap = static_cast<long long>(num_sms) * 8;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

}  // namespace

cudaError_t launch_pack_fwd(const DevSub* subs, const int* col_sub, int C_total, int d_in, int d_out,
                            __nv_bfloat16* at_all, __nv_bfloat16* bt_all, int num_sms, cudaStream_t st, bool pdl) {
  const long long w1 = static_cast<long long>(C_total) * (d_in / 8);
  cudaError_t e = launch_k(k_pack_at, dim3(grid_for(w1, 256, num_sms)), dim3(256), 0, st, pdl, subs, col_sub, C_total,
                           d_in, at_all);
  if (e != cudaSuccess) return e;
  const long long w2 = static_cast<long long>(d_out) * (C_total / 8);
  return launch_k(k_pack_bt, dim3(grid_for(w2, 256, num_sms)), dim3(256), 0, st, pdl, subs, col_sub, C_total, d_out,
                  bt_all);
}

cudaError_t launch_h_images(const DevSeg* segs, const float* col_scale, const MTile* mtiles, const int* img_tile,
                            int n_images, long long N, const float* H, uint8_t* img_out, cudaStream_t st, bool pdl) {
  if (n_images <= 0) return cudaSuccess;
  return launch_k(k_h_images, dim3(n_images), dim3(BM), 0, st, pdl, segs, col_scale, mtiles, img_tile, N, H,
                  img_out);
}

cudaError_t launch_adamw(const AdamItem* items, int n_items, float lr, float beta1, float beta2, float eps,
                         float weight_decay, int step, int num_sms, cudaStream_t st, bool pdl, __nv_bfloat16* at_all,
                         __nv_bfloat16* bt_all, int C_total) {
  if (n_items <= 0) return cudaSuccess;
  const double bc1 = 1.0 - pow(static_cast<double>(beta1), step);
  const double bc2 = 1.0 - pow(static_cast<double>(beta2), step);
  const float decay = 1.0f - lr * weight_decay;
  int grid = n_items;
  if (grid > num_sms * 16) grid = num_sms * 16;
  return launch_k(k_adamw, dim3(grid), dim3(256), 0, st, pdl, items, n_items, lr, beta1, beta2, eps, decay,
                  static_cast<float>(bc1), static_cast<float>(bc2), at_all, bt_all, C_total);
}

}  // namespace mlora
