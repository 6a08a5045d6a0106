// Base GEMMs on CTA pairs with a 4-bit frozen base weight.
//
// "PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §5 and §11.3: a 4-bit
// quantised base (QLoRA) composes with packing.  The pages do not fix the 4-bit format; this
// library reads it as signed 4-bit codes q in [-8, 7] with one fp32 scale per 64 consecutive
// d_in entries of each output column, W[k][o] = q[o][k] * scale[k / 64][o]:
//   Wq     [d_out, d_in / 2] bytes, two codes per byte (even k in the low nibble, two's complement)
//   Wscale [d_in / 64, d_out] fp32 (group-major, so one K slice's scales are contiguous)
//
// The kernel is the bf16 CTA-pair kernel of gemm_2sm.cu with the B operand of the main K loop
// produced in shared memory by four converter warps instead of copied by TMA: the producer
// copies the 4-bit tile and its scales (4.5 KB per CTA per K slice instead of 16 KB), the
// converters expand them to bf16 (round to nearest) in the 128B-swizzled K-major layout the
// MMA reads, fence the writes for the tensor core's async proxy and arrive on the even CTA's
// full barrier.  Forward B rows are output columns (codes read along d_in); backward B rows are
// input columns (codes read across d_out rows, transposed on the way).  The rank term's K slices
// are bf16 and arrive by TMA exactly as in the bf16 kernel.
//
// Roles (320 threads): warp 0 TMA, warp 1 MMA (even CTA), warps 2-5 epilogue, warps 6-9 converters.
#include "common.cuh"
#include "pair.cuh"

namespace mlora {

using namespace pair;

namespace {

constexpr int SW = 5;                          // pipeline stages
constexpr int W4_THREADS = 320;
constexpr int A_BYTES = 128 * BK * 2;          // this CTA's 128 rows of A per stage
constexpr int B_BYTES = 128 * BK * 2;          // this CTA's 128-row half of B per stage (bf16)
constexpr int RAW_BYTES = 128 * BK / 2;        // the same half of B as 4-bit codes
constexpr int SC_BYTES = 128 * 4;              // its scales
constexpr int SMEM_W4 = SW * (A_BYTES + B_BYTES + RAW_BYTES + SC_BYTES) + 1024 + 512;

__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Code e (0..7) of a word whose nibbles were pre-flipped with 0x88888888, as an exact float:
// 2^23 + (nib ^ 8) built by a bit-OR, minus 2^23 + 8, gives the signed code in [-8, 7].
__device__ __forceinline__ float code(uint32_t flipped, int e) {
  return __int_as_float(static_cast<int>(((flipped >> (4 * e)) & 0xFu) | 0x4B000000u)) - 8388616.0f;
}

// Forward: B row n = ct (an output column) = 64 codes along d_in, one scale.
__device__ __forceinline__ void convert_fwd(const uint8_t* raw, const float* sc, uint8_t* b, int ct) {
  const uint4* rp = reinterpret_cast<const uint4*>(raw + ct * 32);
  const uint4 r0 = rp[0], r1 = rp[1];
  const uint32_t w[8] = {r0.x ^ 0x88888888u, r0.y ^ 0x88888888u, r0.z ^ 0x88888888u, r0.w ^ 0x88888888u,
                         r1.x ^ 0x88888888u, r1.y ^ 0x88888888u, r1.z ^ 0x88888888u, r1.w ^ 0x88888888u};
  const float s = sc[ct];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) pk[e / 2] = pack_bf16x2(code(w[c], e) * s, code(w[c], e + 1) * s);
    *reinterpret_cast<uint4*>(b + swz128_offset(ct, 8 * c)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

// Backward: B row n (an input column) = the codes of 64 output rows k at column n, one scale per
// row.  Thread ct converts an 8 (n) x 8 (k) block: n = 8 (ct >> 3) .. +7, k = 8 (ct & 7) .. +7,
// from eight 32-bit loads (8 codes of one k row each), transposed in registers.
__device__ __forceinline__ void convert_bwd(const uint8_t* raw, const float* sc, uint8_t* b, int ct) {
  const int ng = ct >> 3, kg = ct & 7;
  uint32_t wk[8];
  float sk[8];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int k = 8 * kg + kk;
    wk[kk] = *reinterpret_cast<const uint32_t*>(raw + k * 64 + 4 * ng) ^ 0x88888888u;
    sk[kk] = sc[(ng >> 3) * 64 + k];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t pk[4];
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) pk[kk / 2] = pack_bf16x2(code(wk[kk], j) * sk[kk], code(wk[kk + 1], j) * sk[kk + 1]);
    *reinterpret_cast<uint4*>(b + swz128_offset(8 * ng + j, 8 * kg)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

}  // namespace

// tmA: X or dY [N, K] bf16, box (64, 128).  tmQ: Wq bytes, box (32, 128) fwd / (64, 64) bwd.
// tmS: Wscale fp32, box (128, 1) fwd / (64, 2) bwd.  tmE: rank-term B (Bt_all fwd, At_all bwd).
// tmI: staged images, box (64, 128).
template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(W4_THREADS, 1)
    k_gemm_2sm_w4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmE,
                  const __grid_constant__ CUtensorMap tmI, const __grid_constant__ GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + SW * A_BYTES;
  uint8_t* sQ = sB + SW * B_BYTES;
  uint8_t* sS = sQ + SW * RAW_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + SW * SC_BYTES);
  uint64_t* full = bars;               // [SW] (even CTA) A bytes of both CTAs + 8 converter warps + producer
  uint64_t* empty = bars + SW;         // [SW] MMA -> producer and converters of each CTA
  uint64_t* qfull = bars + 2 * SW;     // [SW] this CTA's 4-bit tile and scales -> its converters
  uint64_t* tfull = bars + 3 * SW;     // [2]
  uint64_t* tempty = tfull + 2;        // [2]  (even CTA) both CTAs' epilogues
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1, n_pairs_grid = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(&full[s], 9);   // the even CTA's producer (arrive.expect_tx) + 8 converter warps
      mbar_init(&empty[s], 1);
      mbar_init(&qfull[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmS);
    prefetch_tmap(&tmE);
    prefetch_tmap(&tmI);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const unsigned long long tmo = g.timeout_ns;
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int item = pair_id; ok && item < g.n_items; item += n_pairs_grid) {
        int mp, n;
        decode_pair(g, item, mp, n);
        const int tile = 2 * mp + static_cast<int>(rank);
        const MTile mt = g.mtiles[min(tile, g.n_mtiles - 1)];
        const int m0 = tile * BM;
        const int nh0 = n * BN + static_cast<int>(rank) * 128;
        const int nkb = g.kmain + mt.nch;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
            ok = false;
            break;
          }
          const bool main_part = kb < g.kmain;
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * A_BYTES + (main_part ? 0 : 2 * B_BYTES));
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
          uint8_t* a = sA + stage * A_BYTES;
          if (main_part) {
            tma_load_2d_pair(a, &tmA, bar, kb * BK, m0);
            mbar_arrive_expect_tx(&qfull[stage], RAW_BYTES + SC_BYTES);
            if constexpr (MODE == MODE_FWD) {
              tma_load_2d(sQ + stage * RAW_BYTES, &tmQ, &qfull[stage], kb * (BK / 2), nh0);
              tma_load_2d(sS + stage * SC_BYTES, &tmS, &qfull[stage], nh0, kb);
            } else {
              tma_load_2d(sQ + stage * RAW_BYTES, &tmQ, &qfull[stage], nh0 / 2, kb * BK);
              tma_load_2d(sS + stage * SC_BYTES, &tmS, &qfull[stage], kb * BK, nh0 / 64);
            }
          } else {
            const int e = kb - g.kmain;
            uint8_t* b = sB + stage * B_BYTES;
            tma_load_2d_pair(a, &tmI, bar, 0, (mt.img_off + e) * BM);
            if constexpr (MODE == MODE_FWD) {
              tma_load_2d_pair(b, &tmE, bar, (mt.q_lo + e) * CHUNK_COLS, nh0);
            } else {
              tma_load_2d_pair(b, &tmE, bar, nh0, (mt.q_lo + e) * CHUNK_COLS);
              tma_load_2d_pair(b + 64 * 64 * 2, &tmE, bar, nh0 + 64, (mt.q_lo + e) * CHUNK_COLS);
            }
          }
          if (++stage == SW) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t idesc_k = idesc_bf16(2 * BM, BN, false, false);
      const uint32_t idesc_mn = idesc_bf16(2 * BM, BN, false, true);
      for (int item = pair_id; ok && item < g.n_items; item += n_pairs_grid) {
        int mp, n;
        decode_pair(g, item, mp, n);
        const int nkb = g.kmain + g.mtiles[min(2 * mp, g.n_mtiles - 1)].nch;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_MMA, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, g.err, DEV_ERR_TIMEOUT_MMA, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(sA + stage * A_BYTES);
          const uint32_t b = smem_u32(sB + stage * B_BYTES);
          // main K slices: converted B, K-major; rank-term slices: as in the bf16 kernel
          const bool b_mn = (MODE == MODE_BWD) && kb >= g.kmain;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = smem_desc(a + k * 32, 16, 1024);
            const uint64_t bd = b_mn ? smem_desc(b + k * 2048, 64 * 64 * 2, 1024) : smem_desc(b + k * 32, 16, 1024);
            umma_pair_bf16(d_tmem, ad, bd, b_mn ? idesc_mn : idesc_k, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_pair_commit_mc(&empty[stage], 0x3);
          if (++stage == SW) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_pair_commit_mc(&tfull[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_pair_commit_mc(done, 0x1);
      volatile int no_abort = 0;
      mbar_wait(done, 0, &no_abort, g.err, DEV_ERR_TIMEOUT_TEARDOWN, tmo);
    }
  } else if (warp < 6) {
    const int quarter = warp & 3;
    const int rit = quarter * 32 + lane;
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_leader1 = mapa_shared(smem_u32(&tempty[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(g.out);
    const int ld = g.ld_out;
    for (int item = pair_id; item < g.n_items; item += n_pairs_grid) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, g.err, DEV_ERR_TIMEOUT_EPILOGUE, tmo);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      int mp, n;
      decode_pair(g, item, mp, n);
      const long long row = static_cast<long long>(2 * mp + static_cast<int>(rank)) * BM + rit;
      const int col0 = n * BN;
      const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int cb = 0; cb < BN; cb += 32) {
        uint32_t v[32];
        tmem_ld32(t_acc + cb, v);
        tmem_ld_wait();
        const int col = col0 + cb;
        if (row < g.N && col < ld) {
          __nv_bfloat16* dst = out + row * ld + col;
          if (col + 32 <= ld) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 u;
              u.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
              u.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
              u.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
              u.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
              d4[q] = u;
            }
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u)
              if (col + u < ld) dst[u] = __float2bfloat16_rn(__uint_as_float(v[u]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc ? tempty_leader1 : tempty_leader0);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  } else {
    // converters: 128 threads, thread ct expands row ct of this CTA's B half
    const int ct = threadIdx.x - 192;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t qphase = 0;   // bit s: parity of qfull[s], which completes only on main-K uses of slot s
    bool ok = true;
    for (int item = pair_id; ok && item < g.n_items; item += n_pairs_grid) {
      int mp, n;
      decode_pair(g, item, mp, n);
      const int nkb = g.kmain + g.mtiles[min(2 * mp + static_cast<int>(rank), g.n_mtiles - 1)].nch;
      for (int kb = 0; kb < nkb; ++kb) {
        // the slot is free (MMA done with its previous use) ...
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
          ok = false;
          break;
        }
        if (kb < g.kmain) {
          // ... and its 4-bit tile has landed
          if (!mbar_wait(&qfull[stage], (qphase >> stage) & 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
            ok = false;
            break;
          }
          qphase ^= 1u << stage;
          const uint8_t* raw = sQ + stage * RAW_BYTES;
          const float* sc = reinterpret_cast<const float*>(sS + stage * SC_BYTES);
          uint8_t* b = sB + stage * B_BYTES;
          if constexpr (MODE == MODE_FWD)
            convert_fwd(raw, sc, b, ct);
          else
            convert_bwd(raw, sc, b, ct);
          fence_async_shared();   // generic-proxy writes -> visible to the tensor core
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&full[stage]), 0));
        if (++stage == SW) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }

  if (*abort_flag) {
    const unsigned long long t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 50000ull) {
    }
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int MODE>
cudaError_t launch_gemm_2sm_w4(const CUtensorMap& tmA, const CUtensorMap& tmQ, const CUtensorMap& tmS,
                               const CUtensorMap& tmE, const CUtensorMap& tmI, const GemmArgs& g, int n_pairs,
                               cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_2sm_w4<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_W4);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (g.n_items <= 0) return cudaSuccess;
  return launch_k(k_gemm_2sm_w4<MODE>, dim3(2 * n_pairs), dim3(W4_THREADS), SMEM_W4, stream, g.pdl != 0, tmA, tmQ,
                  tmS, tmE, tmI, g);
}

template cudaError_t launch_gemm_2sm_w4<MODE_FWD>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&, const GemmArgs&, int,
                                                  cudaStream_t);
template cudaError_t launch_gemm_2sm_w4<MODE_BWD>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                  const CUtensorMap&, const CUtensorMap&, const GemmArgs&, int,
                                                  cudaStream_t);

}  // namespace mlora
