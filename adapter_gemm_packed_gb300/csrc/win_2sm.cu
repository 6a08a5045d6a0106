// The memory-bound rank-window products on CTA pairs (tcgen05 cta_group::2, cluster of 2):
//
//   MODE_SHRINK  H_i  = X_i A_i          (+ staged s_i H_i images)
//   MODE_DH      dH_i = s_i dY_i B_i^T   (+ staged dH_i images; "PLoRA: Efficient Concurrent LoRA
//                                         Training for Large Language Models", §9.2 Case 2)
//
// A work item is a 256-token pair of tiles and up to four 64-column chunks of their (shared)
// rank window.  Each CTA streams its own 128 token rows of X (or dY) and holds half of the
// item's chunks of the rank operand (At_all rows K-major for SHRINK, Bt_all MN-major for DH);
// the even CTA issues one M=256 MMA per 16-wide K step over both halves.  Against the
// single-CTA engine (one 128-token tile, two chunks per item) each token re-streams half as
// many bytes of the rank operand from L2, and a tile's X (or dY) is re-read once per four
// chunks instead of once per two: what limits wide windows (jobs with large or several ranks
// sharing a tile).  Items carry an even chunk count (a window of one chunk is padded to two),
// so both CTAs always load whole chunks; a padding chunk is computed and discarded.  Each pair
// runs its own list of items (the planner's per-pair schedule); an item the schedule cuts along
// K runs as pieces on several pairs, each parking fp32 partial sums, and the last piece to
// finish adds them in piece order before writing the outputs.
//
// The epilogue of each CTA writes its own tile: H (SHRINK, fp32) or dH (scaled), and the bf16
// images of s*H / dH per (tile, chunk), zero outside each row's job window, exactly as the
// single-CTA engine does.  Synchronisation follows the CTA-pair GEMM (gemm_2sm.cu).
#include "common.cuh"
#include "pair.cuh"

namespace mlora {

using namespace pair;

namespace {

constexpr int SW2 = 6;                               // pipeline stages
constexpr int WA_BYTES = 128 * BK * 2;               // this CTA's 128 token rows per stage
constexpr int WB_BYTES = 2 * CHUNK_COLS * BK * 2;    // this CTA's <= 2 chunks of the rank operand per stage
constexpr int SMEM_WIN2 = SW2 * (WA_BYTES + WB_BYTES) + 1024 + 256;

__device__ __forceinline__ int find_job(const DevSeg* segs, int first, int last, long long row) {
  int j = first;
  while (j < last && row >= segs[j + 1].off) ++j;
  return j;
}

}  // namespace

// tmA: X [N, d_in] or dY [N, d_out], box (64, 128).  tmB: At_all [C, d_in] box (64, 64) for SHRINK,
// Bt_all [d_out, C] box (64, 64) read MN-major for DH.  g.win: pair items (tile = pair index).
template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    k_win_2sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + SW2 * WA_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + SW2 * WB_BYTES);
  uint64_t* full = bars;               // [SW2] (even CTA) TMA bytes of both CTAs -> MMA
  uint64_t* empty = bars + SW2;        // [SW2] MMA -> each CTA's producer
  uint64_t* tfull = bars + 2 * SW2;    // [2]   MMA -> each CTA's epilogue
  uint64_t* tempty = tfull + 2;        // [2]   (even CTA) both epilogues -> MMA
  uint64_t* done = tempty + 2;         // [1]   (even CTA) MMA drain at teardown
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* ring_hi = tmem_slot + 2;   // (even CTA) ring positions filled, max over both producers

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1, n_pairs_grid = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW2; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
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
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const unsigned long long tmo = g.timeout_ns;
  griddep_wait();
  griddep_launch_dependents();
  // this pair's items: its run of the planner's per-pair list, else every n_pairs_grid-th item
  const int it_first = g.cta_first ? g.cta_first[pair_id] : pair_id;
  const int it_end = g.cta_first ? g.cta_first[pair_id + 1] : g.n_items;
  const int it_step = g.cta_first ? 1 : n_pairs_grid;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_stream = l2_policy_evict_first();
      const uint64_t pol_keep = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0;
      bool ok = true;
      for (int item = it_first; ok && item < it_end; item += it_step) {
        const WinItem w = g.win[item];
        const int m0 = (2 * w.tile + static_cast<int>(rank)) * BM;
        const int nb = w.nq >> 1;                                   // chunks held by this CTA
        const int qb = w.q0 + static_cast<int>(rank) * nb;
        int kb0, nkb;                                               // the item's (or part's) K slices
        win_krange(w, MODE == MODE_DH, g.kmain, kb0, nkb);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (WA_BYTES + nb * CHUNK_COLS * BK * 2));
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
          const int k = kb0 + kb;
          ++filled;
          if (g.debug_drop && leader && pair_id == 0 && filled == 1) {
            // Test hook for the timeout path (see gemm_2sm.cu): armed, nothing copied by this CTA.
          } else {
            tma_load_2d_pair_hint(sA + stage * WA_BYTES, &tmA, bar, k * BK, m0, pol_stream);
            uint8_t* b = sB + stage * WB_BYTES;
            for (int j = 0; j < nb; ++j) {
              if constexpr (MODE == MODE_SHRINK)   // At_all rows (K-major, k = d_in)
                tma_load_2d_pair_hint(b + j * (CHUNK_COLS * BK * 2), &tmB, bar, k * BK, (qb + j) * CHUNK_COLS, pol_keep);
              else                                 // Bt_all [d_out, C] as MN-major (n = rank column, k = d_out)
                tma_load_2d_pair_hint(b + j * (CHUNK_COLS * BK * 2), &tmB, bar, (qb + j) * CHUNK_COLS, k * BK, pol_keep);
            }
          }
          if (++stage == SW2) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      publish_ring_pos(ring_hi, filled);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int item = it_first; ok && item < it_end; item += it_step) {
        const WinItem w = g.win[item];
        int kb0, nkb;
        win_krange(w, MODE == MODE_DH, g.kmain, kb0, nkb);
        const uint32_t idesc = idesc_bf16(2 * BM, w.nq * CHUNK_COLS, false, MODE == MODE_DH);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_MMA, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 256;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, g.err, DEV_ERR_TIMEOUT_MMA, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(sA + stage * WA_BYTES);
          const uint32_t b = smem_u32(sB + stage * WB_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = smem_desc(a + k * 32, 16, 1024);
            const uint64_t bd = (MODE == MODE_DH) ? smem_desc(b + k * 2048, CHUNK_COLS * BK * 2, 1024)
                                                  : smem_desc(b + k * 32, 16, 1024);
            umma_pair_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_pair_commit_mc(&empty[stage], 0x3);
          if (++stage == SW2) {
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
  } else {
    const int quarter = warp & 3;
    const int rit = quarter * 32 + lane;   // accumulator row (TMEM lane) owned by this thread
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_leader1 = mapa_shared(smem_u32(&tempty[1]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int item = it_first; item < it_end; item += it_step) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, g.err, DEV_ERR_TIMEOUT_EPILOGUE, tmo);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const WinItem w = g.win[item];
      const int tile = 2 * w.tile + static_cast<int>(rank);
      bool released = false;   // this warp has handed the accumulator back to the MMA
      if (tile < g.n_mtiles) {   // an odd last tile has no partner: its half computed zeros
        const MTile mt = g.mtiles[tile];
        const long long row = static_cast<long long>(tile) * BM + rit;
        int j = -1;
        if (row < g.N) j = find_job(g.segs, mt.seg_first, mt.seg_last, row);
        long long hbase = 0;
        int c_lo = 0, c_hi = 0;
        float s = 0.f;
        if (j >= 0) {
          const DevSeg sg = g.segs[j];
          c_lo = sg.c;
          c_hi = sg.c + sg.r;
          s = sg.s;
          hbase = sg.h_off + (row - sg.off) * sg.r - sg.c;
        }
        const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * 256;
        // One chunk's 64 accumulated columns of this thread's row -> H (SHRINK: H = acc) or dH
        // (DH: dH = s*acc), and the bf16 image s*acc, zero outside the row's job window.
        auto emit_chunk = [&](int jq, const uint32_t* vv) {
          const int q = w.q0 + jq;
          uint8_t* img = g.img_out + static_cast<size_t>(mt.img_off + q - mt.q_lo) * IMG_BYTES;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t* v = vv + half * 32;
            const int cbase = q * CHUNK_COLS + half * 32;
            uint32_t pk[16];
#pragma unroll
            for (int u = 0; u < 32; u += 4) {
              const int c0 = cbase + u;
              float a[4];
              bool in[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                a[k] = __uint_as_float(v[u + k]);
                in[k] = c0 + k >= c_lo && c0 + k < c_hi;
              }
              // the scale of each column's adapter (one per job unless the pack shares its input)
              float sk[4] = {s, s, s, s};
              if (g.col_scale) {
#pragma unroll
                for (int k = 0; k < 4; ++k) sk[k] = __ldg(g.col_scale + c0 + k);
              }
              float hv[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) hv[k] = (MODE == MODE_SHRINK) ? a[k] : sk[k] * a[k];
              float* hp = g.hout + hbase + c0;
              if (in[0] && in[3] && ((reinterpret_cast<uintptr_t>(hp) & 15u) == 0)) {
                *reinterpret_cast<float4*>(hp) = make_float4(hv[0], hv[1], hv[2], hv[3]);
              } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  if (in[k]) hp[k] = hv[k];
              }
              pk[u / 2] = pack_bf16x2(in[0] ? sk[0] * a[0] : 0.f, in[1] ? sk[1] * a[1] : 0.f);
              pk[u / 2 + 1] = pack_bf16x2(in[2] ? sk[2] * a[2] : 0.f, in[3] ? sk[3] * a[3] : 0.f);
            }
            uint4* dst = reinterpret_cast<uint4*>(img + rit * (CHUNK_COLS * 2) + half * 64);
#pragma unroll
            for (int k16 = 0; k16 < 4; ++k16)
              dst[k16] = make_uint4(pk[4 * k16], pk[4 * k16 + 1], pk[4 * k16 + 2], pk[4 * k16 + 3]);
          }
        };
        const int nreal = min(w.nq, mt.q_lo + mt.nch - w.q0);   // chunks past the window are padding
        if (w.nparts == 1) {
#pragma unroll 1
          for (int jq = 0; jq < nreal; ++jq) {
            uint32_t vv[64];
            tmem_ld32(t_acc + jq * CHUNK_COLS, *reinterpret_cast<uint32_t(*)[32]>(&vv[0]));
            tmem_ld32(t_acc + jq * CHUNK_COLS + 32, *reinterpret_cast<uint32_t(*)[32]>(&vv[32]));
            tmem_ld_wait();
            emit_chunk(jq, vv);
          }
        } else {
          // A part of an item cut along K: park this part's sums ([pbase + part][CTA][256 columns]
          // [128 rows], fp32, so that a warp's 32 rows of one column are one 128-byte line), hand
          // the accumulator back, and count the arrival of this warp's 32 rows.  The last of the
          // item's parts to arrive reads all parts' sums back in part order (a fixed order:
          // results do not depend on timing) and writes the item's outputs.  Nothing waits for
          // another CTA.
          const size_t stride = static_cast<size_t>(BM) * 256;
          float* mine = g.partials + (static_cast<size_t>(w.pbase + w.part) * 2 + rank) * stride + rit;
#pragma unroll 1
          for (int jq = 0; jq < nreal; ++jq) {
            uint32_t vv[64];
            tmem_ld32(t_acc + jq * CHUNK_COLS, *reinterpret_cast<uint32_t(*)[32]>(&vv[0]));
            tmem_ld32(t_acc + jq * CHUNK_COLS + 32, *reinterpret_cast<uint32_t(*)[32]>(&vv[32]));
            tmem_ld_wait();
            float* col = mine + static_cast<size_t>(jq * CHUNK_COLS) * BM;
#pragma unroll
            for (int c = 0; c < 64; ++c) col[c * BM] = __uint_as_float(vv[c]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acc ? tempty_leader1 : tempty_leader0);
          released = true;
          __threadfence();   // this warp's sums are visible before its arrival is counted
          __syncwarp();
          int last = 0;
          if (lane == 0) {
            int* cnt = g.part_cnt + (w.slot * 2 + static_cast<int>(rank)) * 4 + quarter;
            if (atomicAdd(cnt, 1) == w.nparts - 1) {
              *cnt = 0;       // every part has arrived: ready for the next launch
              last = 1;
            }
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            __threadfence();
            const float* base = g.partials + (static_cast<size_t>(w.pbase) * 2 + rank) * stride + rit;
#pragma unroll 1
            for (int jq = 0; jq < nreal; ++jq) {
              const float* col = base + static_cast<size_t>(jq * CHUNK_COLS) * BM;
              // part by part, all 64 columns' loads of a part in flight together; each column is
              // summed in part order
              float acc_v[64];
#pragma unroll 1
              for (int p = 0; p < w.nparts; ++p) {
                const float* src = col + p * 2 * stride;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                  const float x = __ldcg(src + c * BM);
                  acc_v[c] = p ? acc_v[c] + x : x;
                }
              }
              uint32_t vv[64];
#pragma unroll
              for (int c = 0; c < 64; ++c) vv[c] = __float_as_uint(acc_v[c]);
              emit_chunk(jq, vv);
            }
          }
        }
      }
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(acc ? tempty_leader1 : tempty_leader0);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // No copy is issued after this barrier; the even CTA then waits for the last ring positions'
  // copies (both CTAs') to land, and the odd CTA's shared memory stays alive until it has.
  tc_fence_before();
  cluster_sync_all();
  if (leader && threadIdx.x == 0) drain_ring<SW2>(full, *reinterpret_cast<volatile uint32_t*>(ring_hi), g.err, tmo);
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int MODE>
cudaError_t launch_win_2sm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& g, int n_pairs,
                           cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = ensure_smem_attr(k_win_2sm<MODE>, SMEM_WIN2, attr_done);
  if (e != cudaSuccess) return e;
  if (g.n_items <= 0) return cudaSuccess;
  return launch_k(k_win_2sm<MODE>, dim3(2 * n_pairs), dim3(GEMM_THREADS), SMEM_WIN2, stream, g.pdl != 0, tmA, tmB, g);
}

template cudaError_t launch_win_2sm<MODE_SHRINK>(const CUtensorMap&, const CUtensorMap&, const GemmArgs&, int,
                                                 cudaStream_t);
template cudaError_t launch_win_2sm<MODE_DH>(const CUtensorMap&, const CUtensorMap&, const GemmArgs&, int,
                                             cudaStream_t);

}  // namespace mlora
