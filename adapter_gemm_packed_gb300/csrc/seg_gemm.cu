// Segmented tensor-core GEMM engine for the packed LoRA layer (sm_103a: tcgen05 + TMEM + TMA).
//
// One persistent, warp-specialised kernel template computes the products of the layer on
// single CTAs ("PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §9.2: tiles
// run along the token and hidden dimensions, never along the rank).  The base GEMMs run on CTA
// pairs by default (gemm_2sm.cu; this engine's FWD/BWD with MLORA_GEMM_SINGLE_CTA), and shrink /
// dH move to CTA pairs for wide rank windows (win_2sm.cu):
//
//   MODE_FWD    Y  = X W + s_i H_i B_i        base GEMM; the rank term is appended as extra
//                                              K slices of the same TMEM accumulator
//                                              ([X | Htilde] x [Wt | Bt_all]^T)
//   MODE_BWD    dX = dY W^T + dH_i A_i^T      same, W (from Wt) and A (from At_all) read MN-major
//   MODE_SHRINK H_i = X_i A_i                  per tile, N = the tile's rank window
//   MODE_DH     dH_i = s_i dY_i B_i^T          per tile, N = the tile's rank window (Case 2),
//                                              B read MN-major from Bt_all
//   MODE_DA     dA_i = X_i^T dH_i              token reduction (Case 3)
//   MODE_DB     dB_i = s_i H_i^T dY_i          token reduction (Case 1)
//
// The packed rank space: job i owns columns [c_i, c_i + rp_i) (rp_i = r_i rounded up to 16),
// cut into 64-column chunks.  A 128-token tile that covers jobs i1..im needs only the chunks
// spanning their windows.  Htilde / dHtilde are kept as "staged images": for each (tile,
// chunk) a row-major [128 x 64] bf16 block (TMA applies the 128B swizzle on the way into shared
// memory), holding s_j H_j (resp. dH_j) in the rows of job j and the columns of job j, and zero
// everywhere else.  The
// zeros make the rank-term K extension of FWD/BWD and the token reductions of DA/DB exact
// per job without masks in the main loop (tLoRA's "adaptively reconstructed low-rank tiles",
// read as tiles assembled from the jobs a token tile happens to cover).
//
// Roles (192 threads, 320 for dA / dB; one CTA per SM, persistent over a static work list):
//   warp 0     TMA producer (one lane) into a STAGES-deep smem ring
//   warp 1     TMEM allocator and MMA issuer (one lane), two 256-column accumulators
//   warps 2-5  epilogue: TMEM -> registers -> global (lane quarter = warp id % 4); dA / dB have
//              warps 2-9, two per lane quarter (one per 128-row half of the item)
// The CTA-pair base GEMMs (gemm_2sm.cu) write Y / dX through shared memory and TMA stores; this
// engine's single-CTA base GEMMs (kept for comparison) store from registers.
// Every wait is bounded (see mbar_wait): on expiry the CTA records a status code, drains
// what it issued, frees TMEM and returns.
#include "common.cuh"

namespace mlora {

namespace {

// Shared-memory ring geometry per mode.  The tensor-bound single-CTA base GEMMs stage 16 KB of
// A and 32 KB of B per K slice (4 stages).  The memory-bound modes stream one operand from HBM
// (X or dY, 16 KB per slice, loaded with an evict-first L2 policy) against a small operand that
// many CTAs re-read from L2 (up to two 64-column rank chunks, <= 16 KB, evict-last): six stages
// keep 96 KB of the streamed operand in flight per SM (a bare TMA streaming loop on a GB300
// reaches 6.6 TB/s with 4 x 16 KB per SM).
// dA / dB items cover 256 rows of d_in / d_out (two M = 128 MMAs per K step sharing one staged
// image operand), so their ring holds 32 KB of the streamed operand per stage.
// dB's epilogue also stages each warp's 32 rows x 16 columns in shared memory to store dB^T rows
// with consecutive lanes on consecutive addresses: a row's four float4 sit at slots k ^ ((row >> 1)
// & 3), so that both the row-wise writes (one row per lane) and the reads (eight rows of 16
// columns per instruction) touch every bank once per 128 bytes.
constexpr int DB_STAGE_FLOATS = 32 * 16;
__device__ __forceinline__ int db_slot(int row, int k) { return row * 4 + (k ^ ((row >> 1) & 3)); }

// dA / dB run two epilogue warps per TMEM lane quarter (one per 128-row half of the item): their
// items are a few K slices long and their epilogue writes as many bytes as the item reads, so its
// latency chain (TMEM load, staging, store) would otherwise set the pace.
template <int MODE>
struct Ring {
  static constexpr bool kBase = MODE == MODE_FWD || MODE == MODE_BWD;
  static constexpr bool kWgrad = MODE == MODE_DA || MODE == MODE_DB;
  static constexpr int kStages = kBase ? 4 : (kWgrad ? 4 : 6);
  static constexpr int kABytes = kWgrad ? 2 * A_STAGE_BYTES : A_STAGE_BYTES;
  static constexpr int kBBytes = kBase ? B_STAGE_BYTES : MAX_ITEM_CHUNKS * CHUNK_COLS * BK * 2;
  static constexpr int kEpiWarps = kWgrad ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kStageBytes = MODE == MODE_DB ? kEpiWarps * DB_STAGE_FLOATS * 4 : 0;
  static constexpr int kSmem = kStages * (kABytes + kBBytes) + 1024 + 256 + kStageBytes;
};
static_assert(Ring<MODE_DB>::kSmem <= 232448, "dB ring + staging exceed the shared memory of a CTA");

// The CTA's items: a contiguous run of the planner's per-CTA schedule (dA / dB), else every
// gridDim.x-th item from blockIdx.x.
struct ItemRange {
  int first, end, step;
};
__device__ __forceinline__ ItemRange item_range(const GemmArgs& g) {
  if (g.cta_first) return ItemRange{g.cta_first[blockIdx.x], g.cta_first[blockIdx.x + 1], 1};
  return ItemRange{static_cast<int>(blockIdx.x), g.n_items, static_cast<int>(gridDim.x)};
}

__device__ __forceinline__ void decode_mn(const GemmArgs& g, int item, int& m, int& n) {
  const int per_group = g.group_m * g.n_tiles_n;
  const int group = item / per_group;
  const int first_m = group * g.group_m;
  const int gm = min(g.group_m, g.n_mtiles - first_m);
  const int in_group = item - group * per_group;
  m = first_m + in_group % gm;
  n = in_group / gm;
}

// K slices and accumulator columns (MMA N) of a base-GEMM or rank-window item (dA / dB items
// carry both in their descriptor, which the roles read one item ahead).
template <int MODE>
__device__ __forceinline__ int item_kblocks(const GemmArgs& g, int item) {
  if constexpr (MODE == MODE_FWD || MODE == MODE_BWD) {
    int m, n;
    decode_mn(g, item, m, n);
    return g.kmain + g.mtiles[m].nch;
  } else if constexpr (MODE == MODE_SHRINK) {
    return g.kmain;
  } else {
    return g.win[item].dh_nkb;
  }
}

template <int MODE>
__device__ __forceinline__ int item_ncols(const GemmArgs& g, int item) {
  if constexpr (MODE == MODE_FWD || MODE == MODE_BWD) {
    return BN;
  } else {
    return CHUNK_COLS * g.win[item].nq;
  }
}

// ------------------------------------------------------------------- producer (one thread)
template <int MODE>
__device__ __forceinline__ void produce_kblock(const GemmArgs& g, const CUtensorMap* tmA, const CUtensorMap* tmB,
                                               const CUtensorMap* tmE, const CUtensorMap* tmI, int item, int kb,
                                               uint8_t* sA, uint8_t* sB, uint64_t* full, uint64_t pol_stream,
                                               uint64_t pol_keep) {
  if constexpr (MODE == MODE_FWD || MODE == MODE_BWD) {
    int m, n;
    decode_mn(g, item, m, n);
    const int m0 = m * BM, n0 = n * BN;
    mbar_arrive_expect_tx(full, A_STAGE_BYTES + B_STAGE_BYTES);
    if (kb < g.kmain) {
      tma_load_2d(sA, tmA, full, kb * BK, m0);
      if constexpr (MODE == MODE_FWD) {
        tma_load_2d(sB, tmB, full, kb * BK, n0);
      } else {
        // W as the B operand of dX = dY W^T: element (n = d_in index, k = d_out index) is
        // Wt[k][n], contiguous along n -> four 64-wide MN-major boxes.
#pragma unroll
        for (int j = 0; j < 4; ++j) tma_load_2d(sB + j * (BK * 64 * 2), tmB, full, n0 + 64 * j, kb * BK);
      }
    } else {
      const MTile mt = g.mtiles[m];
      const int e = kb - g.kmain;
      tma_load_2d(sA, tmI, full, 0, (mt.img_off + e) * BM);          // staged image, [128 x 64]
      if constexpr (MODE == MODE_FWD) {
        tma_load_2d(sB, tmE, full, (mt.q_lo + e) * CHUNK_COLS, n0);  // Bt_all rows, K-major
      } else {
        // At_all [C, d_in] as the MN-major B operand (n = d_in index, k = rank column)
#pragma unroll
        for (int j = 0; j < 4; ++j) tma_load_2d(sB + j * (BK * 64 * 2), tmE, full, n0 + 64 * j, (mt.q_lo + e) * CHUNK_COLS);
      }
    }
  } else if constexpr (MODE == MODE_SHRINK || MODE == MODE_DH) {
    const WinItem w = g.win[item];
    const int m0 = w.tile * BM;
    const int k = (MODE == MODE_DH) ? w.dh_kb0 + kb : kb;   // dH: only the covered d_out slices
    mbar_arrive_expect_tx(full, A_STAGE_BYTES + w.nq * (CHUNK_COLS * BK * 2));
    tma_load_2d_hint(sA, tmA, full, k * BK, m0, pol_stream);
    for (int j = 0; j < w.nq; ++j) {
      if constexpr (MODE == MODE_SHRINK)   // At_all rows (K-major, k = d_in)
        tma_load_2d_hint(sB + j * (CHUNK_COLS * BK * 2), tmB, full, k * BK, (w.q0 + j) * CHUNK_COLS, pol_keep);
      else                                 // Bt_all [d_out, C] as MN-major (n = rank column, k = d_out)
        tma_load_2d_hint(sB + j * (CHUNK_COLS * BK * 2), tmB, full, (w.q0 + j) * CHUNK_COLS, k * BK, pol_keep);
    }
  }
}

// dA / dB: the K slice of 64-token half-tile gh of item w (mt: the descriptor of gh's 128-token tile).
__device__ __forceinline__ void produce_wgrad(const CUtensorMap* tmA, const CUtensorMap* tmI, const WItem& w,
                                              const MTile& mt, int gh, uint8_t* sA, uint8_t* sB, uint64_t* full,
                                              uint64_t pol_stream, uint64_t pol_keep) {
  const int h = gh & 1;
  mbar_arrive_expect_tx(full, 2 * A_STAGE_BYTES + w.nq * (IMG_BYTES / 2));
  // X (dA) or dY (dB) as an MN-major operand: 64 hidden columns x 64 tokens per box, four boxes
  // for the item's 256 rows (two M = 128 operands, 16 KB each)
#pragma unroll
  for (int j = 0; j < 4; ++j) tma_load_2d_hint(sA + j * (64 * 64 * 2), tmA, full, w.row0 + 64 * j, gh * 64, pol_stream);
  // staged images as an MN-major operand: 64 rank columns x 64 tokens per box
  for (int j = 0; j < w.nq; ++j)
    tma_load_2d_hint(sB + j * (IMG_BYTES / 2), tmI, full, 0, (mt.img_off + w.q0 + j - mt.q_lo) * BM + h * 64,
                     pol_keep);
}

// ------------------------------------------------------------------- MMA (one thread)
template <int MODE>
__device__ __forceinline__ void mma_kblock(const GemmArgs& g, int item, int kb, uint32_t sA, uint32_t sB,
                                           uint32_t d_tmem, int ncols) {
  if constexpr (MODE == MODE_FWD || MODE == MODE_BWD) {
    const bool b_mn = MODE == MODE_BWD;   // W and At_all are both read MN-major by the backward
    const uint32_t idesc = idesc_bf16(BM, BN, false, b_mn);
#pragma unroll
    for (int k = 0; k < BK / 16; ++k) {
      const uint64_t a = smem_desc(sA + k * 32, 16, 1024);
      const uint64_t b = b_mn ? smem_desc(sB + k * 2048, 64 * 64 * 2, 1024) : smem_desc(sB + k * 32, 16, 1024);
      umma_bf16(d_tmem, a, b, idesc, (kb > 0 || k > 0) ? 1u : 0u);
    }
  } else if constexpr (MODE == MODE_SHRINK || MODE == MODE_DH) {
    constexpr bool b_mn = MODE == MODE_DH;
    const uint32_t idesc = idesc_bf16(BM, ncols, false, b_mn);
#pragma unroll
    for (int k = 0; k < BK / 16; ++k) {
      const uint64_t b = b_mn ? smem_desc(sB + k * 2048, CHUNK_COLS * BK * 2, 1024) : smem_desc(sB + k * 32, 16, 1024);
      umma_bf16(d_tmem, smem_desc(sA + k * 32, 16, 1024), b, idesc, (kb > 0 || k > 0) ? 1u : 0u);
    }
  } else {
    // two 128-row halves of the item into accumulator columns [0, N) and [128, 128 + N)
    const uint32_t idesc = idesc_bf16(BM, ncols, true, true);
#pragma unroll
    for (int k = 0; k < BK / 16; ++k) {
      const uint64_t b = smem_desc(sB + k * 2048, IMG_BYTES / 2, 1024);
      umma_bf16(d_tmem, smem_desc(sA + k * 2048, 64 * 64 * 2, 1024), b, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      umma_bf16(d_tmem + 128, smem_desc(sA + A_STAGE_BYTES + k * 2048, 64 * 64 * 2, 1024), b, idesc,
                (kb > 0 || k > 0) ? 1u : 0u);
    }
  }
}

// ------------------------------------------------------------------- epilogues (128 threads)
__device__ __forceinline__ int find_seg(const DevSeg* segs, int first, int last, long long row) {
  int j = first;
  while (j < last && row >= segs[j + 1].off) ++j;
  return j;
}

// Write columns [32 h, 32 h + 32) of chunk jq of a dA / dB item's row half mh: this thread's
// row, values v.  All 32 lanes of the warp call it together (the dB store is warp-cooperative).
template <int MODE>
__device__ __forceinline__ void wgrad_emit(const GemmArgs& g, const WItem& w, int mh, int jq, int h,
                                           const uint32_t (&v)[32], float* stage, int quarter, int lane) {
  const int bound = (MODE == MODE_DA) ? g.d_in : g.d_out;
  const int row = w.row0 + mh * BM + quarter * 32 + lane;   // d_in (DA) or d_out (DB) index
  const int cfirst = (w.q0 + jq) * CHUNK_COLS + h * 32;      // packed column of v[0]
  const int t0 = cfirst - w.c0;                              // rank index of v[0]
  if (g.subs) {
    // several adapters per job (one per projection): each adapter of this item's job takes
    // its own run of the chunk's columns (dB only for the output rows its B covers).  A chunk
    // can also hold other jobs' columns; this item reduced over its own job's tokens only,
    // so those are left to the other jobs' items.
    if (row >= bound) return;
#pragma unroll 1
    for (int a = w.seg * g.n_groups; a < (w.seg + 1) * g.n_groups; ++a) {
      const DevSub sb = g.subs[a];
      const int lo = max(sb.c0, cfirst), hi = min(sb.c0 + sb.r, cfirst + 32);
      if (lo >= hi) continue;
      if constexpr (MODE == MODE_DA) {
        // dAt[t][row]: for a fixed t the 32 lanes write 32 consecutive rows (coalesced)
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int c = cfirst + u;
          if (c >= lo && c < hi) sb.dAt[static_cast<size_t>(c - sb.c0) * g.d_in + row] = __uint_as_float(v[u]);
        }
      } else {
        if (row < sb.o_lo || row >= sb.o_hi) continue;
        // dBt[row - o_lo][t]: one contiguous run per thread, 16-byte stores where aligned
        float* dst = sb.dBt + static_cast<size_t>(row - sb.o_lo) * sb.r + (cfirst - sb.c0);   // + u
        const bool al = ((static_cast<long long>(row - sb.o_lo) * sb.r + (cfirst - sb.c0)) & 3) == 0;
#pragma unroll
        for (int u = 0; u < 32; u += 4) {
          const int c = cfirst + u;
          if (al && c >= lo && c + 3 < hi) {
            *reinterpret_cast<float4*>(dst + u) = make_float4(__uint_as_float(v[u]), __uint_as_float(v[u + 1]),
                                                              __uint_as_float(v[u + 2]), __uint_as_float(v[u + 3]));
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (c + k >= lo && c + k < hi) dst[u + k] = __uint_as_float(v[u + k]);
          }
        }
      }
    }
    return;
  }
  if constexpr (MODE == MODE_DA) {
    // dAt_i[t][row]: for a fixed t the 32 lanes write 32 consecutive rows (coalesced)
    if (row >= bound) return;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int t = t0 + u;
      if (t >= 0 && t < w.r) w.out[static_cast<size_t>(t) * g.d_in + row] = __uint_as_float(v[u]);
    }
  } else {
    // dBt_i[row][t]: a thread holds one row, but a row's values are contiguous in memory, so the
    // warp goes through shared memory and stores along the rows instead, 16 columns at a time
    const int r = w.r;
    const int row_w = w.row0 + mh * BM + quarter * 32;   // the warp's first row
    const int nrows = min(32, bound - row_w);            // its rows inside d_out
    if (nrows <= 0) return;                              // the same for the whole warp
    float* buf = stage;
    float4* buf4 = reinterpret_cast<float4*>(stage);
    const bool al4 = (r & 3) == 0 && (reinterpret_cast<uintptr_t>(w.out) & 15) == 0;
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      const int tq = t0 + qq * 16;   // rank index of this quarter's first column
      const int lo = max(0, tq), hi = min(r, tq + 16);
      if (hi <= lo) continue;        // the same for the whole warp
      if (lo == 0 && hi == r && r < 16) {
        // every row's r values lie in these 16 columns: the warp's rows are one contiguous run of
        // 32 r floats, packed densely here and stored by consecutive lanes
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (tq + u >= 0 && tq + u < r) buf[lane * r + tq + u] = __uint_as_float(v[qq * 16 + u]);
        __syncwarp();
        float* dst = w.out + static_cast<size_t>(row_w) * r;
        for (int e = lane; e < nrows * r; e += 32) dst[e] = buf[e];
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          buf4[db_slot(lane, k)] = make_float4(__uint_as_float(v[qq * 16 + 4 * k]), __uint_as_float(v[qq * 16 + 4 * k + 1]),
                                               __uint_as_float(v[qq * 16 + 4 * k + 2]),
                                               __uint_as_float(v[qq * 16 + 4 * k + 3]));
        __syncwarp();
        if (al4 && lo == tq && hi == tq + 16) {
          // eight rows of 16 columns per store instruction, 16 bytes per lane
#pragma unroll
          for (int it = 0; it < 4; ++it) {
            const int rr = it * 8 + (lane >> 2), k = lane & 3;
            if (rr < nrows)
              *reinterpret_cast<float4*>(w.out + static_cast<size_t>(row_w + rr) * r + tq + 4 * k) = buf4[db_slot(rr, k)];
          }
        } else {
          // rows not 16-byte aligned (r not a multiple of 4) or part of the 16 columns: the wq valid
          // columns of the warp's rows taken in row order, element e at row e / wq and column
          // lo + e % wq, 32 consecutive elements per store instruction (one run of wq floats per row)
          const int wq = hi - lo, n_el = nrows * wq;
          const int step_r = 32 / wq, step_c = 32 - step_r * wq;
          int rr = lane / wq, c = lane - rr * wq;
          for (int e = lane; e < n_el; e += 32) {
            const int cq = lo - tq + c;   // column within the staged 16
            w.out[static_cast<size_t>(row_w + rr) * r + lo + c] = buf[db_slot(rr, cq >> 2) * 4 + (cq & 3)];
            rr += step_r;
            c += step_c;
            if (c >= wq) {
              c -= wq;
              ++rr;
            }
          }
        }
      }
      __syncwarp();   // the staging is reused next
    }
  }
}

// Epilogue of a base-GEMM or rank-window item (the accumulator is handed back by the caller).
template <int MODE>
__device__ __forceinline__ bool epilogue_item(const GemmArgs& g, int item, uint32_t t_acc, int quarter, int lane) {
  const int rit = quarter * 32 + lane;   // accumulator row owned by this thread
  if constexpr (MODE == MODE_FWD || MODE == MODE_BWD) {
    int m, n;
    decode_mn(g, item, m, n);
    const long long row = static_cast<long long>(m) * BM + rit;
    const int col0 = n * BN;
    const int ld = g.ld_out;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(g.out);
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
  } else if constexpr (MODE == MODE_SHRINK || MODE == MODE_DH) {
    const WinItem w = g.win[item];
    const MTile mt = g.mtiles[w.tile];
    const long long row = static_cast<long long>(w.tile) * BM + rit;
    int j = -1;
    if (row < g.N) j = find_seg(g.segs, mt.seg_first, mt.seg_last, row);
    long long hbase = 0;
    int c_lo = 0, c_hi = 0, r = 1;
    float s = 0.f;
    if (j >= 0) {
      const DevSeg sg = g.segs[j];
      r = sg.r;
      c_lo = sg.c;
      c_hi = sg.c + sg.r;
      s = sg.s;
      hbase = sg.h_off + (row - sg.off) * sg.r - sg.c;
    }
    // SHRINK: H = acc, image = s*acc.  DH: dH = s*acc, image = s*acc.
#pragma unroll 1
    for (int jq = 0; jq < w.nq; ++jq) {
      const int q = w.q0 + jq;
      uint8_t* img = g.img_out + static_cast<size_t>(mt.img_off + q - mt.q_lo) * IMG_BYTES;
      uint32_t vv[64];
      tmem_ld32(t_acc + jq * CHUNK_COLS, *reinterpret_cast<uint32_t(*)[32]>(&vv[0]));
      tmem_ld32(t_acc + jq * CHUNK_COLS + 32, *reinterpret_cast<uint32_t(*)[32]>(&vv[32]));
      tmem_ld_wait();
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
          // H / dH row segment: one 16-byte store when the four columns are in the window and aligned
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
    }
  }
  return false;
}

// dA / dB epilogue of item w (read ahead by the caller; it carries its job's window and output, so
// no dependent load sits between two items).  Returns true if it already handed the accumulator
// back (arrived on tempty_bar).
template <int MODE>
// This warp handles row half mh of the item (lanes of its quarter); `stage` is its own staging.
__device__ __forceinline__ bool epilogue_wgrad(const GemmArgs& g, const WItem& w, uint32_t t_acc,
                                               int quarter, int mh, int lane, float* stage, uint64_t* tempty_bar) {
  const int rit = quarter * 32 + lane;   // accumulator row owned by this thread
  if (w.nparts == 1) {
#pragma unroll 1
    for (int jq = 0; jq < w.nq; ++jq) {
      // both 32-column halves of the chunk in flight before one wait
      uint32_t v[64];
      tmem_ld32(t_acc + mh * 128 + jq * CHUNK_COLS, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(t_acc + mh * 128 + jq * CHUNK_COLS + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      wgrad_emit<MODE>(g, w, mh, jq, 0, *reinterpret_cast<const uint32_t(*)[32]>(&v[0]), stage, quarter, lane);
      wgrad_emit<MODE>(g, w, mh, jq, 1, *reinterpret_cast<const uint32_t(*)[32]>(&v[32]), stage, quarter, lane);
    }
    return false;
  }
  // One part of an item cut across CTAs: park this part's sums, hand the accumulator back, count
  // the arrival; the last part of the item to arrive sums all parts in part order and writes the
  // gradient.  No CTA waits on another.  A part parks each 32-column group (row half mh, chunk jq,
  // half h) that holds some of the job's columns as 8 runs of 4 columns, a run being [128 rows] of
  // float4: a warp's 32 rows of a run are one 512-byte line, and the last part's sum has 8 loads
  // in flight per part, two parts per round trip.
  auto live = [&](int jq, int h) {
    const int t0 = (w.q0 + jq) * CHUNK_COLS + h * 32 - w.c0;
    return max(0, t0) < min(w.r, t0 + 32);
  };
  float4* base = reinterpret_cast<float4*>(g.partials + static_cast<size_t>(w.pbase) * WG_UNIT);
  const size_t part_f4 = static_cast<size_t>(w.nq) * (WG_UNIT / 4);   // float4s per part
  float4* mine = base + static_cast<size_t>(w.part) * part_f4;
#pragma unroll 1
  for (int jq = 0; jq < w.nq; ++jq) {
    if (!live(jq, 0) && !live(jq, 1)) continue;   // the same for the whole warp
    uint32_t v[64];
    tmem_ld32(t_acc + mh * 128 + jq * CHUNK_COLS, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
    tmem_ld32(t_acc + mh * 128 + jq * CHUNK_COLS + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (!live(jq, h)) continue;
      float4* dst = mine + static_cast<size_t>(((mh * w.nq + jq) * 2 + h) * 8) * BM + rit;
#pragma unroll
      for (int u4 = 0; u4 < 8; ++u4)
        dst[u4 * BM] = make_float4(__uint_as_float(v[h * 32 + 4 * u4]), __uint_as_float(v[h * 32 + 4 * u4 + 1]),
                                   __uint_as_float(v[h * 32 + 4 * u4 + 2]), __uint_as_float(v[h * 32 + 4 * u4 + 3]));
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(tempty_bar);
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    __threadfence();   // the warp's stores (ordered before this by the warp barrier) before the count
    int* cnt = g.part_cnt + w.cnt * 8 + quarter * 2 + mh;
    last = atomicAdd(cnt, 1) == w.nparts - 1;
    if (last) *cnt = 0;   // every part has arrived: the counter is ready for the next launch
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return true;
  __threadfence();
  const int S = w.nparts;
#pragma unroll 1
  for (int jq = 0; jq < w.nq; ++jq)
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      if (!live(jq, h)) continue;
      const float4* src = base + static_cast<size_t>(((mh * w.nq + jq) * 2 + h) * 8) * BM + rit;
      float4 acc[8];
#pragma unroll 1
      for (int p = 0; p < S; p += 2) {
        float4 a[8], b[8];
        const bool two = p + 1 < S;
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4) {
          a[u4] = __ldcg(src + p * part_f4 + u4 * BM);
          if (two) b[u4] = __ldcg(src + (p + 1) * part_f4 + u4 * BM);
        }
#pragma unroll
        for (int u4 = 0; u4 < 8; ++u4) {
          if (p == 0) {
            acc[u4] = a[u4];
          } else {
            acc[u4].x += a[u4].x;
            acc[u4].y += a[u4].y;
            acc[u4].z += a[u4].z;
            acc[u4].w += a[u4].w;
          }
          if (two) {
            acc[u4].x += b[u4].x;
            acc[u4].y += b[u4].y;
            acc[u4].z += b[u4].z;
            acc[u4].w += b[u4].w;
          }
        }
      }
      uint32_t v[32];
#pragma unroll
      for (int u4 = 0; u4 < 8; ++u4) {
        v[4 * u4] = __float_as_uint(acc[u4].x);
        v[4 * u4 + 1] = __float_as_uint(acc[u4].y);
        v[4 * u4 + 2] = __float_as_uint(acc[u4].z);
        v[4 * u4 + 3] = __float_as_uint(acc[u4].w);
      }
      wgrad_emit<MODE>(g, w, mh, jq, h, v, stage, quarter, lane);
    }
  return true;
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(Ring<MODE>::kThreads, 1)
    k_seg_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmI,
               const __grid_constant__ GemmArgs g) {
  constexpr int STAGES = Ring<MODE>::kStages;
  constexpr int A_BYTES = Ring<MODE>::kABytes;
  constexpr int B_BYTES = Ring<MODE>::kBBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint64_t* full = bars;                 // [STAGES]  TMA -> MMA
  uint64_t* empty = bars + STAGES;       // [STAGES]  MMA -> TMA
  uint64_t* tfull = bars + 2 * STAGES;   // [2]       MMA -> epilogue
  uint64_t* tempty = tfull + 2;          // [2]       epilogue -> MMA
  uint64_t* done = tempty + 2;           // [1]       MMA drain at teardown
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* stage_buf = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);   // dB epilogue staging

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ItemRange items = item_range(g);
  constexpr bool kWgrad = Ring<MODE>::kWgrad;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], Ring<MODE>::kEpiWarps);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmE);
    prefetch_tmap(&tmI);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const unsigned long long tmo = g.timeout_ns;
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_stream = l2_policy_evict_first();
      const uint64_t pol_keep = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // dA / dB items are a few K slices long: the next item's descriptor and its first tile's
      // record are read one item ahead, and each further tile's record one tile ahead, so no
      // dependent load sits between two copies
      WItem w{};
      MTile mt_first{};
      if (kWgrad && items.first < items.end) {
        w = g.witems[items.first];
        mt_first = g.mtiles[w.ga >> 1];
      }
      for (int item = items.first; ok && item < items.end; item += items.step) {
        WItem w_next{};
        if (kWgrad && item + items.step < items.end) w_next = g.witems[item + items.step];
        int nkb;
        if constexpr (kWgrad) nkb = w.gb - w.ga;
        else nkb = item_kblocks<MODE>(g, item);
        int t_have = w.ga >> 1;
        MTile mt = mt_first, mt_ahead{};
        if (kWgrad && ((w.gb - 1) >> 1) > t_have) mt_ahead = g.mtiles[t_have + 1];
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_PRODUCER, tmo)) {
            ok = false;
            break;
          }
          if (g.debug_drop && blockIdx.x == 0 && issued == 0) {
            // Test hook for the timeout path: arm the slot, issue nothing.  The MMA warp's
            // bounded wait on it runs out and records a status code; nothing faults or hangs.
            mbar_arrive_expect_tx(&full[stage], A_BYTES);
          } else if constexpr (kWgrad) {
            const int gh = w.ga + kb;   // 64-token half-tile
            if ((gh >> 1) != t_have) {  // the next tile (half-tiles run in order)
              t_have = gh >> 1;
              mt = mt_ahead;
              if (((w.gb - 1) >> 1) > t_have) mt_ahead = g.mtiles[t_have + 1];
            }
            produce_wgrad(&tmA, &tmI, w, mt, gh, sA + stage * A_BYTES, sB + stage * B_BYTES, &full[stage], pol_stream,
                          pol_keep);
          } else {
            produce_kblock<MODE>(g, &tmA, &tmB, &tmE, &tmI, item, kb, sA + stage * A_BYTES, sB + stage * B_BYTES,
                                 &full[stage], pol_stream, pol_keep);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (kWgrad && item + items.step < items.end) mt_first = g.mtiles[w_next.ga >> 1];
        w = w_next;
      }
      if (!ok || *abort_flag) {
        // Drain: wait (bounded) for the copies of the last STAGES issued slots to land so
        // no bulk copy is still writing this CTA's shared memory when it exits.
        volatile int no_abort = 0;
        for (int k = 0; k < STAGES && k < issued; ++k) {
          if (--stage < 0) {
            stage = STAGES - 1;
            phase ^= 1u;
          }
          mbar_wait(&full[stage], phase, &no_abort, g.err, DEV_ERR_TIMEOUT_TEARDOWN, tmo);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      WItem w{};
      if (kWgrad && items.first < items.end) w = g.witems[items.first];
      for (int item = items.first; ok && item < items.end; item += items.step) {
        WItem w_next{};
        if (kWgrad && item + items.step < items.end) w_next = g.witems[item + items.step];
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, g.err, DEV_ERR_TIMEOUT_MMA, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        int nkb, ncols;
        if constexpr (kWgrad) {
          nkb = w.gb - w.ga;
          ncols = CHUNK_COLS * w.nq;
        } else {
          nkb = item_kblocks<MODE>(g, item);
          ncols = item_ncols<MODE>(g, item);
        }
        w = w_next;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, g.err, DEV_ERR_TIMEOUT_MMA, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_kblock<MODE>(g, item, kb, smem_u32(sA + stage * A_BYTES), smem_u32(sB + stage * B_BYTES), d_tmem,
                           ncols);
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA issued by this thread has completed once `done` flips.
      umma_commit(done);
      volatile int no_abort = 0;
      mbar_wait(done, 0, &no_abort, g.err, DEV_ERR_TIMEOUT_TEARDOWN, tmo);
    }
  } else {
    const int quarter = warp & 3;
    const int mh = (warp - 2) >> 2;   // dA / dB: the item's row half this warp writes
    float* my_stage = stage_buf + (warp - 2) * DB_STAGE_FLOATS;
    int acc = 0;
    uint32_t acc_phase = 0;
    // dA / dB: the next item's descriptor (which carries its job's window and output) is read as
    // soon as this item's epilogue is done, while the MMA may still be working on the next
    // accumulator
    WItem w{};
    if (kWgrad && items.first < items.end) w = g.witems[items.first];
    for (int item = items.first; item < items.end; item += items.step) {
      // One lane waits; the warp follows its decision so the .sync.aligned TMEM loads below
      // are always executed by all 32 lanes together.
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, g.err, DEV_ERR_TIMEOUT_EPILOGUE, tmo);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      bool released;
      if constexpr (kWgrad)
        released = epilogue_wgrad<MODE>(g, w, t_acc, quarter, mh, lane, my_stage, &tempty[acc]);
      else
        released = epilogue_item<MODE>(g, item, t_acc, quarter, lane);
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      }
      if (kWgrad && item + items.step < items.end) w = g.witems[item + items.step];   // ahead of the next wait
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Host-side launch helper (one per mode).
template <int MODE>
cudaError_t launch_seg_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmE,
                            const CUtensorMap& tmI, const GemmArgs& g, int grid, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = ensure_smem_attr(k_seg_gemm<MODE>, Ring<MODE>::kSmem, attr_done);
  if (e != cudaSuccess) return e;
  if (g.n_items <= 0) return cudaSuccess;
  return launch_k(k_seg_gemm<MODE>, dim3(grid), dim3(Ring<MODE>::kThreads), Ring<MODE>::kSmem, stream, g.pdl != 0, tmA, tmB,
                  tmE, tmI, g);
}

template cudaError_t launch_seg_gemm<MODE_FWD>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_seg_gemm<MODE_BWD>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_seg_gemm<MODE_SHRINK>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const CUtensorMap&, const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_seg_gemm<MODE_DH>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const CUtensorMap&, const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_seg_gemm<MODE_DA>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const CUtensorMap&, const GemmArgs&, int, cudaStream_t);
template cudaError_t launch_seg_gemm<MODE_DB>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const CUtensorMap&, const GemmArgs&, int, cudaStream_t);

}  // namespace mlora
