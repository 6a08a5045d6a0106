// Base GEMMs on CTA pairs that expand a 4-bit frozen base weight in shared memory (the
// MLORA_W4_FUSED variant; by default the library expands the weight once per call with
// w4_expand.cu and runs the bf16 GEMMs, which is faster at training batch sizes because this
// kernel repeats the expansion for every 256-token tile pair).
//
// "PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §5 and §11.3: a 4-bit
// quantised base (QLoRA) composes with packing.  The pages do not fix the 4-bit format; this
// library reads it as signed 4-bit codes q in [-8, 7] with one fp32 scale per 64 consecutive
// d_in entries of each output column, W[k][o] = q[o][k] * scale[k / 64][o]:
//   Wq     [d_out, d_in / 2] bytes, two codes per byte (even k in the low nibble, two's complement)
//   Wscale [d_in / 64, d_out] fp32 (group-major, so one K slice's scales are contiguous)
//
// The kernel is the bf16 CTA-pair kernel of gemm_2sm.cu with the B operand of the main K loop
// produced in shared memory by eight converter warps instead of copied by TMA.  A separate
// producer warp copies the 4-bit tiles and their scales (4.5 KB per CTA per K slice instead of
// 16 KB) into an 8-slot ring of their own, so those copies run ahead of the MMA.  A converter
// warp expands its share of a tile into registers (bf16, round to nearest) before the slot of
// the main ring is free, then only stores it, fences the writes for the tensor core's async
// proxy and signals the even CTA's full barrier with a 16-byte bulk copy (its transaction bytes
// are part of the barrier's expected count; a cluster-scope release arrive would put a memory
// barrier on the converters' serial path).  Forward B rows are output columns and the codes run
// along them (K-major B); backward B is read MN-major, so the codes of one d_out row, which
// run along d_in, land in place without a transpose.  The rank term's K slices are bf16 and
// arrive by TMA exactly as in the bf16 kernel.
//
// Roles (480 threads): warp 0 TMA for A (and the rank term), warp 1 MMA (even CTA), warps 2-5
// epilogue, warps 6-13 converters, warp 14 TMA for the 4-bit tiles.
#include "common.cuh"
#include "pair.cuh"
#include "w4.cuh"

namespace mlora {

using namespace pair;
using w4::expand8;

namespace {

constexpr int SW = 5;                          // main ring stages (A and bf16 B)
constexpr int RW = 8;                          // 4-bit ring stages
constexpr int N_CONV_WARPS = 8;
constexpr int W4_THREADS = 32 * (7 + N_CONV_WARPS);
constexpr int RAWP_WARP = 6 + N_CONV_WARPS;    // the 4-bit tile producer
constexpr int A_BYTES = 128 * BK * 2;          // this CTA's 128 rows of A per stage
constexpr int B_BYTES = 128 * BK * 2;          // this CTA's 128-row half of B per stage (bf16)
constexpr int RAW_BYTES = 128 * BK / 2;        // the same half of B as 4-bit codes
constexpr int SC_BYTES = 128 * 4;              // its scales
constexpr int SIG_BYTES = 16;                  // one converter warp's ready signal
constexpr int N_SIG = 2 * N_CONV_WARPS;        // signals per stage (both CTAs)
constexpr int BAR_AREA = 2048;
constexpr int SMEM_W4 = SW * (A_BYTES + B_BYTES) + RW * (RAW_BYTES + SC_BYTES) + BAR_AREA + 1024;

__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One converter thread's share of a K slice: 32 codes, as four 16-byte bf16 groups.
struct Share {
  uint4 v[4];
};

// Forward: B row n (an output column) holds 64 codes along d_in with one scale.  Thread ct
// (0..255) takes half a row: n = ct / 2, codes 32 (ct % 2) .. +31 (one 16-byte load; a warp
// reads 512 contiguous bytes).
__device__ __forceinline__ void expand_fwd(const uint8_t* raw, const float* sc, int ct, uint64_t magic2, Share& o) {
  const uint4 w = *reinterpret_cast<const uint4*>(raw + ct * 16);
  const float s = sc[ct >> 1];
  o.v[0] = expand8(w.x, s, magic2);
  o.v[1] = expand8(w.y, s, magic2);
  o.v[2] = expand8(w.z, s, magic2);
  o.v[3] = expand8(w.w, s, magic2);
}

__device__ __forceinline__ void store_fwd(uint8_t* b, int ct, const Share& o) {
  const int n = ct >> 1, c0 = 4 * (ct & 1);
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(b + swz128_offset(n, 8 * (c0 + j))) = o.v[j];
}

// Backward: row k of the tile (a d_out row, K of dX = dY W^T) holds 128 codes along d_in (N);
// scale (n / 64, k).  Word L = 256 j + ct (j = 0..3) is codes n = 8 (L % 16) .. +7 of row
// k = L / 16; it lands, still in n order, in the MN-major 128B-swizzled layout: 64-wide n
// blocks 8 KB apart, one 128-byte line per k.
__device__ __forceinline__ void expand_bwd(const uint8_t* raw, const float* sc, int ct, uint64_t magic2, Share& o) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int L = 256 * j + ct;
    const int k = L >> 4, ng = L & 15;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(raw + 4 * L);
    o.v[j] = expand8(w, sc[(ng >> 3) * 64 + k], magic2);
  }
}

__device__ __forceinline__ void store_bwd(uint8_t* b, int ct, const Share& o) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int L = 256 * j + ct;
    const int k = L >> 4, ng = L & 15;
    *reinterpret_cast<uint4*>(b + (ng >> 3) * 8192 + swz128_offset(k, 8 * (ng & 7))) = o.v[j];
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
  uint8_t* sS = sQ + RW * RAW_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + RW * SC_BYTES);
  uint64_t* full = bars;               // [SW] (even CTA) producer + A bytes of both CTAs + warp signals
  uint64_t* empty = full + SW;         // [SW] MMA -> producer and converters of each CTA
  uint64_t* qfull = empty + SW;        // [RW] this CTA's 4-bit tile and scales -> its converters
  uint64_t* qempty = qfull + RW;       // [RW] this CTA's converter warps -> the 4-bit producer
  uint64_t* tfull = qempty + RW;       // [2]
  uint64_t* tempty = tfull + 2;        // [2]  (even CTA) both CTAs' epilogues
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* ring_hi = tmem_slot + 2;   // (even CTA) main-ring positions filled, max over every issuer
  uint8_t* sig_dst = reinterpret_cast<uint8_t*>(bars) + 1024;    // [N_SIG][16] (even CTA) signal landing slots
  uint8_t* sig_src = sig_dst + N_SIG * SIG_BYTES;               // [16] this CTA's signal payload

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1, n_pairs_grid = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's producer (arrive.expect_tx); the rest is bytes
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < RW; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], N_CONV_WARPS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *ring_hi = 0;
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
      uint32_t filled = 0;
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
          if (leader)
            mbar_arrive_expect_tx(&full[stage], 2 * A_BYTES + (main_part ? 0 : 2 * B_BYTES) + N_SIG * SIG_BYTES);
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
          uint8_t* a = sA + stage * A_BYTES;
          ++filled;
          if (main_part) {
            tma_load_2d_pair(a, &tmA, bar, kb * BK, m0);
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
      publish_ring_pos(ring_hi, filled);
    }
  } else if (warp == RAWP_WARP) {
    if (lane == 0) {
      // the 4-bit tiles of every main K slice, in the order the converters take them
      const uint64_t keep = l2_policy_evict_last();
      int rs = 0;
      uint32_t rphase = 0;
      uint32_t rfilled = 0;
      bool ok = true;
      for (int item = pair_id; ok && item < g.n_items; item += n_pairs_grid) {
        int mp, n;
        decode_pair(g, item, mp, n);
        const int nh0 = n * BN + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < g.kmain; ++kb) {
          if (!mbar_wait(&qempty[rs], rphase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&qfull[rs], RAW_BYTES + SC_BYTES);
          ++rfilled;
          if constexpr (MODE == MODE_FWD) {
            tma_load_2d_hint(sQ + rs * RAW_BYTES, &tmQ, &qfull[rs], kb * (BK / 2), nh0, keep);
            tma_load_2d_hint(sS + rs * SC_BYTES, &tmS, &qfull[rs], nh0, kb, keep);
          } else {
            tma_load_2d_hint(sQ + rs * RAW_BYTES, &tmQ, &qfull[rs], nh0 / 2, kb * BK, keep);
            tma_load_2d_hint(sS + rs * SC_BYTES, &tmS, &qfull[rs], kb * BK, nh0 / 64, keep);
          }
          if (++rs == RW) {
            rs = 0;
            rphase ^= 1u;
          }
        }
      }
      // This CTA's own ring: slot p % RW was re-filled only after the converters released it, so
      // the copies of every position but the last RW have landed; wait (bounded) for those.
      volatile int no_abort = 0;
      for (uint32_t p = rfilled > RW ? rfilled - RW : 0; p < rfilled; ++p)
        if (!mbar_wait(&qfull[p % RW], (p / RW) & 1u, &no_abort, g.err, DEV_ERR_TIMEOUT_TEARDOWN, tmo)) break;
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // backward B is MN-major throughout (converted W^T slices and the rank term alike)
      const uint32_t idesc = idesc_bf16(2 * BM, BN, false, MODE == MODE_BWD);
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
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = smem_desc(a + k * 32, 16, 1024);
            const uint64_t bd = MODE == MODE_BWD ? smem_desc(b + k * 2048, 64 * 64 * 2, 1024)
                                                 : smem_desc(b + k * 32, 16, 1024);
            umma_pair_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
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
    // converters: 256 threads; every K slice of the main ring gets one signal per warp
    const int ct = threadIdx.x - 192;
    const int cw = ct >> 5;
    const uint32_t my_sig = mapa_shared(smem_u32(sig_dst + (N_CONV_WARPS * static_cast<int>(rank) + cw) * SIG_BYTES), 0);
    const uint64_t magic2 = w4::magic_pair();
    int stage = 0, rs = 0;
    uint32_t phase = 0, rphase = 0;
    uint32_t filled = 0;
    bool ok = true;
    for (int item = pair_id; ok && item < g.n_items; item += n_pairs_grid) {
      int mp, n;
      decode_pair(g, item, mp, n);
      const int nkb = g.kmain + g.mtiles[min(2 * mp + static_cast<int>(rank), g.n_mtiles - 1)].nch;
      for (int kb = 0; kb < nkb; ++kb) {
        const bool main_part = kb < g.kmain;
        Share sh;
        if (main_part) {
          // expand this share of the 4-bit tile into registers and hand its slot back ...
          if (!mbar_wait(&qfull[rs], rphase, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
            ok = false;
            break;
          }
          const uint8_t* raw = sQ + rs * RAW_BYTES;
          const float* sc = reinterpret_cast<const float*>(sS + rs * SC_BYTES);
          if constexpr (MODE == MODE_FWD)
            expand_fwd(raw, sc, ct, magic2, sh);
          else
            expand_bwd(raw, sc, ct, magic2, sh);
          __syncwarp();
          if (lane == 0) mbar_arrive(&qempty[rs]);
          if (++rs == RW) {
            rs = 0;
            rphase ^= 1u;
          }
        }
        // ... then wait for the main ring's slot (the MMA done with its previous use)
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
          ok = false;
          break;
        }
        if (main_part) {
          uint8_t* b = sB + stage * B_BYTES;
          if constexpr (MODE == MODE_FWD)
            store_fwd(b, ct, sh);
          else
            store_bwd(b, ct, sh);
          fence_async_shared();   // generic-proxy writes -> visible to the tensor core
        }
        __syncwarp();
        if (lane == 0) bulk_signal_remote(my_sig, sig_src, mapa_shared(smem_u32(&full[stage]), 0));
        ++filled;
        if (++stage == SW) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0) publish_ring_pos(ring_hi, filled);
  }

  // No copy or signal is issued after this barrier; the even CTA then waits for the last main-ring
  // positions (both CTAs' copies and converter signals) to land, and the odd CTA's shared memory
  // stays alive until it has.
  tc_fence_before();
  cluster_sync_all();
  if (leader && threadIdx.x == 0) drain_ring<SW>(full, *reinterpret_cast<volatile uint32_t*>(ring_hi), g.err, tmo);
  __syncwarp();
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
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = ensure_smem_attr(k_gemm_2sm_w4<MODE>, SMEM_W4, attr_done);
  if (e != cudaSuccess) return e;
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
