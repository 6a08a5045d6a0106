// Base GEMMs of the packed LoRA layer on CTA pairs (tcgen05 cta_group::2, cluster of 2).
//
//   MODE_FWD  Y  = X W + s_i H_i B_i      ([X | Htilde] x [Wt | Bt_all]^T, one accumulator)
//   MODE_BWD  dX = dY W^T + dH_i A_i^T    ([dY | dHtilde] x [W | A]^T, W and A read MN-major from
//                                         Wt and At_all)
//
// A pair of CTAs on the two SMs of a TPC computes one 256-token x 256-column tile: each CTA
// stages its own 128 rows of A and its own 128-row half of B per 64-wide K slice (32 KB); a ring
// slot holds two such slices (64 KB per CTA, three slots), and the even CTA issues one M=256,
// N=256 tcgen05.mma per 16-wide K step that reads both CTAs' shared memory and writes each CTA's
// 128 accumulator lanes.  Against the single-CTA 128x256 tile this halves the B bytes each SM
// pulls from L2 per FLOP (the single-CTA kernel's profile showed the tensor pipe waiting on
// operands at ~60 % activity with L2 and DRAM far from saturated).  Two slices per slot halve
// the barrier waits, slot releases and copy arms per MMA against one slice per slot (six slots
// of 32 KB): the layer's GEMMs measured 3-6 % faster with the same bytes in flight.
//
// Synchronisation: the even CTA's full[s] barrier collects the TMA bytes of both CTAs (the odd
// CTA's copies signal it through .cta_group::2); the MMA warp's commits are multicast to both
// CTAs' empty[s] / tfull[a]; both CTAs' epilogue warps arrive on the even CTA's tempty[a].
// The rank term's K extension is identical for both halves because the planner gives both
// 128-token tiles of a pair the union of their rank-chunk ranges.
// Tail: when the last wave of 256x256 tiles would fill at most half of the CTA pairs, the planner
// splits those tiles into two 256x128 halves (items from g.n_full_items on), so the last wave
// takes half the time; a half tile's MMA has N = 128 and each CTA loads 64 rows of its B.
// Every wait is bounded (mbar_wait); on expiry the CTA records a status code and unwinds.
#include "common.cuh"
#include "pair.cuh"

namespace mlora {

using namespace pair;

namespace {

constexpr int S2 = 3;                         // pipeline stages, two 64-wide K slices each
constexpr int A2_BYTES = 128 * BK * 2;        // this CTA's 128 rows of A per K slice
constexpr int B2_BYTES = 128 * BK * 2;        // this CTA's 128-row half of B per K slice
constexpr int STAGE_A = 2 * A2_BYTES, STAGE_B = 2 * B2_BYTES;
constexpr int Y_CHUNK_BYTES = BM * 64 * 2;    // one staged 128-row x 64-column bf16 output box
// ring, then barriers (a 1 KB slot, so the staging that follows stays 1 KB aligned for its
// 128-byte swizzle), two output boxes, and slack to align the dynamic base
constexpr int SMEM_2SM = S2 * (STAGE_A + STAGE_B) + 1024 + 2 * Y_CHUNK_BYTES + 1024;
constexpr int EPI_BAR = 1;                    // named barrier of the four epilogue warps
constexpr int EPI_ISSUER = 64;                // thread that issues the epilogue's TMA stores

}  // namespace

// tmB / tmE: 128-row boxes for the forward's K-major B halves; tmB64 / tmE64: the same tensors
// with 64-row boxes (half tiles).  The backward's MN-major B uses 64-wide boxes throughout.
// tmY: the output (Y or dX), 64-column x 128-row boxes, 128-byte swizzle.
template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_2sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmI,
               const __grid_constant__ CUtensorMap tmB64, const __grid_constant__ CUtensorMap tmE64,
               const __grid_constant__ CUtensorMap tmY, const __grid_constant__ GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S2 * STAGE_A;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S2 * STAGE_B);
  uint64_t* full = bars;               // [S2]  (even CTA) TMA bytes of both CTAs -> MMA
  uint64_t* empty = bars + S2;         // [S2]  MMA -> each CTA's producer
  uint64_t* tfull = bars + 2 * S2;     // [2]   MMA -> each CTA's epilogue
  uint64_t* tempty = tfull + 2;        // [2]   (even CTA) both epilogues -> MMA
  uint64_t* done = tempty + 2;         // [1]   (even CTA) MMA drain at teardown
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* ring_hi = tmem_slot + 2;   // (even CTA) ring positions filled, max over both producers
  uint8_t* ystage = reinterpret_cast<uint8_t*>(bars) + 1024;   // [2] staged output boxes

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs_grid = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S2; ++s) {
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
    prefetch_tmap(&tmE);
    prefetch_tmap(&tmI);
    prefetch_tmap(&tmY);
    if (MODE == MODE_FWD && g.n_full_items < g.n_items) {
      prefetch_tmap(&tmB64);
      prefetch_tmap(&tmE64);
    }
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
      for (int item = pair; ok && item < g.n_items; item += n_pairs_grid) {
        int mp, col0, width;
        decode_item(g, item, mp, col0, width);
        const bool half = width < BN;
        const int tile = 2 * mp + static_cast<int>(rank);
        const MTile mt = g.mtiles[min(tile, g.n_mtiles - 1)];   // a missing odd tile borrows its partner's
        const int m0 = tile * BM;
        const int nh0 = col0 + static_cast<int>(rank) * (width / 2);   // this CTA's half of the item's columns
        const int nkb = g.kmain + mt.nch;
        for (int kb0 = 0; kb0 < nkb; kb0 += 2) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
            ok = false;
            break;
          }
          const int nsub = nkb - kb0 < 2 ? nkb - kb0 : 2;
          if (leader) mbar_arrive_expect_tx(&full[stage], nsub * 2 * (A2_BYTES + width * BK));
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
          ++filled;
          for (int h = 0; h < nsub; ++h) {
            const int kb = kb0 + h;
            uint8_t* a = sA + stage * STAGE_A + h * A2_BYTES;
            uint8_t* b = sB + stage * STAGE_B + h * B2_BYTES;
            if (g.debug_drop && leader && pair == 0 && filled == 1) {
              // Test hook for the timeout path: the slot is armed for both CTAs' bytes but this
              // CTA copies nothing into it, so the MMA's bounded wait runs out and records a status
              // code; the teardown drain then waits out the peer's copies.  Nothing faults or hangs.
            } else if (kb < g.kmain) {
              tma_load_2d_pair(a, &tmA, bar, kb * BK, m0);
              if constexpr (MODE == MODE_FWD) {
                tma_load_2d_pair(b, half ? &tmB64 : &tmB, bar, kb * BK, nh0);
              } else {
                tma_load_2d_pair(b, &tmB, bar, nh0, kb * BK);
                if (!half) tma_load_2d_pair(b + 64 * 64 * 2, &tmB, bar, nh0 + 64, kb * BK);
              }
            } else {
              const int e = kb - g.kmain;
              tma_load_2d_pair(a, &tmI, bar, 0, (mt.img_off + e) * BM);
              if constexpr (MODE == MODE_FWD) {
                tma_load_2d_pair(b, half ? &tmE64 : &tmE, bar, (mt.q_lo + e) * CHUNK_COLS, nh0);
              } else {
                tma_load_2d_pair(b, &tmE, bar, nh0, (mt.q_lo + e) * CHUNK_COLS);
                if (!half) tma_load_2d_pair(b + 64 * 64 * 2, &tmE, bar, nh0 + 64, (mt.q_lo + e) * CHUNK_COLS);
              }
            }
          }
          if (++stage == S2) {
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
      for (int item = pair; ok && item < g.n_items; item += n_pairs_grid) {
        int mp, col0, width;
        decode_item(g, item, mp, col0, width);
        const uint32_t idesc = idesc_bf16(2 * BM, width, false, MODE == MODE_BWD);
        const int nkb = g.kmain + g.mtiles[min(2 * mp, g.n_mtiles - 1)].nch;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_MMA, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb0 = 0; kb0 < nkb; kb0 += 2) {
          if (!mbar_wait(&full[stage], phase, abort_flag, g.err, DEV_ERR_TIMEOUT_MMA, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = nkb - kb0 < 2 ? nkb - kb0 : 2;
          constexpr bool b_mn = MODE == MODE_BWD;   // W and At_all are both read MN-major
          for (int h = 0; h < nsub; ++h) {
            const uint32_t a = smem_u32(sA + stage * STAGE_A + h * A2_BYTES);
            const uint32_t b = smem_u32(sB + stage * STAGE_B + h * B2_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t ad = smem_desc(a + k * 32, 16, 1024);
              const uint64_t bd = b_mn ? smem_desc(b + k * 2048, 64 * 64 * 2, 1024) : smem_desc(b + k * 32, 16, 1024);
              umma_pair_bf16(d_tmem, ad, bd, idesc, (kb0 + h > 0 || k > 0) ? 1u : 0u);
            }
          }
          umma_pair_commit_mc(&empty[stage], 0x3);
          if (++stage == S2) {
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
    // Epilogue: per 64-column chunk of the tile, TMEM -> registers -> bf16 -> a staged box in
    // shared memory (128-byte swizzle: row r's 16-byte piece j at slot j ^ (r & 7)) -> one TMA
    // store of 128 rows x 64 columns.  Whole 128-byte rows reach the L2 instead of 16-byte pieces of
    // 32 rows per store instruction.  Two staged boxes alternate; a box is rewritten only after the
    // store that read it two chunks earlier has finished reading.  The four warps take every
    // decision together (named barrier EPI_BAR), so none can leave the others waiting at it.
    const int quarter = warp & 3;
    const int rit = quarter * 32 + lane;
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_leader1 = mapa_shared(smem_u32(&tempty[1]), 0);
    const bool issuer = threadIdx.x == EPI_ISSUER;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t chunk_no = 0;
    const int ld = g.ld_out;
    for (int item = pair; item < g.n_items; item += n_pairs_grid) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, g.err, DEV_ERR_TIMEOUT_EPILOGUE, tmo);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!named_bar_and(EPI_BAR, 128, ok)) break;
      tc_fence_after();
      int mp, col0, width;
      decode_item(g, item, mp, col0, width);
      const int m0 = (2 * mp + static_cast<int>(rank)) * BM;   // this CTA's first output row
      const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      const int n_chunks = width / 64;
#pragma unroll 1
      for (int c = 0; c < n_chunks; ++c, ++chunk_no) {
        uint32_t v[64];
        tmem_ld32(t_acc + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(t_acc + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        if (c == n_chunks - 1) {   // the accumulator is read: hand it back to the MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acc ? tempty_leader1 : tempty_leader0);
        }
        uint4 u[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          u[j].x = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
          u[j].y = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
          u[j].z = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
          u[j].w = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
        }
        uint8_t* box = ystage + (chunk_no & 1u) * Y_CHUNK_BYTES;
        if (issuer) bulk_wait_group_read<1>();   // the store of two chunks ago has read this box
        named_bar_sync(EPI_BAR, 128);
        uint8_t* row_base = box + rit * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(row_base + ((j ^ (rit & 7)) << 4)) = u[j];
        fence_proxy_async_smem();
        named_bar_sync(EPI_BAR, 128);
        if (issuer) {
          const int col = col0 + c * 64;
          if (m0 < g.N && col < ld) tma_store_2d(&tmY, box, col, m0);
          bulk_commit_group();   // one group per chunk, empty when nothing was stored
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (issuer) bulk_wait_group<0>();   // every store written before the CTA leaves
  }

  // No copy is issued after this barrier; the even CTA then waits for the last ring positions'
  // copies (both CTAs') to land, and the odd CTA's shared memory stays alive until it has.
  tc_fence_before();
  cluster_sync_all();
  if (leader && threadIdx.x == 0) drain_ring<S2>(full, *reinterpret_cast<volatile uint32_t*>(ring_hi), g.err, tmo);
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int MODE>
cudaError_t launch_gemm_2sm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmE,
                            const CUtensorMap& tmI, const CUtensorMap& tmB64, const CUtensorMap& tmE64,
                            const CUtensorMap& tmY, const GemmArgs& g, int n_pairs, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = ensure_smem_attr(k_gemm_2sm<MODE>, SMEM_2SM, attr_done);
  if (e != cudaSuccess) return e;
  if (g.n_items <= 0) return cudaSuccess;
  return launch_k(k_gemm_2sm<MODE>, dim3(2 * n_pairs), dim3(GEMM_THREADS), SMEM_2SM, stream, g.pdl != 0, tmA, tmB,
                  tmE, tmI, tmB64, tmE64, tmY, g);
}

template cudaError_t launch_gemm_2sm<MODE_FWD>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_gemm_2sm<MODE_BWD>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const GemmArgs&, int, cudaStream_t);

}  // namespace mlora
