// Internal definitions shared by the CUDA translation units of the packed LoRA library:
// device-side tables built by the planner, kernel argument blocks, and thin inline-PTX
// wrappers for the sm_103a features the kernels use (tcgen05 MMA/TMEM, TMA bulk tensor
// copies, mbarriers).
#pragma once
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace mlora {

// ---------------------------------------------------------------------------------------
// Tiling constants of the segmented tensor-core GEMM engine.
// A 128-row tile of tokens (or of d_in/d_out rows for the weight-gradient products) is the
// M side of every tcgen05 MMA; operands move in 64-element (128-byte) K slices, so every
// smem operand tile is a stack of 128B-swizzled 8-row atoms (1024 bytes each).
// ---------------------------------------------------------------------------------------
constexpr int BM = 128;              // MMA M (rows of the accumulator = TMEM lanes)
constexpr int BN = 256;              // max MMA N (accumulator columns per buffer)
constexpr int BK = 64;               // K slice per pipeline stage (64 bf16 = 128 bytes)
constexpr int A_STAGE_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_STAGE_BYTES = BN * BK * 2;       // 32 KB
constexpr int CHUNK_COLS = 64;       // rank-window chunk: 64 packed rank columns
constexpr int IMG_BYTES = BM * CHUNK_COLS * 2;   // one staged [128 x 64] bf16 image (16 KB)
constexpr int RANK_PAD = 16;         // each job's rank window is padded to a multiple of 16
constexpr int GEMM_THREADS = 192;    // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int TMEM_COLS = 512;       // two 256-column fp32 accumulators
constexpr int MAX_ITEM_CHUNKS = 2;  // rank chunks per shrink / dH / dA / dB work item (N <= 128)

enum GemmMode : int {
  MODE_FWD = 0,     // Y  = X  Wt^T + Htilde  Bt_all^T          (rank term as extra K slices)
  MODE_BWD = 1,     // dX = dY W    + dHtilde A_all^T           (W read MN-major from Wt)
  MODE_SHRINK = 2,  // H  = X  At_all^T over the tile's rank window -> H (fp32) + Htilde images
  MODE_DH = 3,      // dH = s dY B_all^T over the tile's rank window -> dH (fp32) + dHtilde images
  MODE_DA = 4,      // dA = X^T dHtilde  (token reduction, both operands MN-major)
  MODE_DB = 5       // dB = dY^T Htilde  (token reduction, both operands MN-major)
};

// Per-job record on the device.
struct DevSeg {
  long long off;       // first token row
  int n;               // tokens
  int r;               // rank
  int c;               // first column of the job's window in the packed rank space
  int rp;              // padded window width (multiple of RANK_PAD)
  float s;             // scale alpha / r
  int pad0;
  long long h_off;     // element offset of the job's [n, r] block in H / dH
  float* At;
  float* Bt;
  float* dAt;
  float* dBt;
};

// One adapter of a job (a job has one per projection of a shared-input pack, else one): its
// ranks occupy the packed columns [c0, c0 + r) of the job's window, its B covers the output
// columns [o_lo, o_hi) (B^T is [o_hi - o_lo, r]).
struct DevSub {
  float* At;
  float* Bt;
  float* dAt;
  float* dBt;
  int c0;
  int r;
  int o_lo, o_hi;
  float s;
  int job;
  int pad0, pad1;
};

// Per 128-token tile: which jobs it covers and where its staged rank images live.
struct MTile {
  int seg_first, seg_last;   // jobs overlapping the tile (inclusive)
  int q_lo, nch;             // 64-column chunks [q_lo, q_lo + nch) of the packed rank space
  int img_off;               // index of the tile's first staged image
  int pad0, pad1, pad2;
};

// Rank-window work item (shrink / dH): one tile, up to MAX_ITEM_CHUNKS chunks.
struct WinItem {
  int tile, q0, nq;
  int dh_kb0, dh_nkb;   // dH: the 64-wide d_out slices its chunks' adapters cover (all of d_out
                        // unless the pack shares its input across projections)
  // The CTA-pair schedule can cut an item along K into `nparts` pieces on different pairs: piece
  // `part` covers the share [f0, f1) / WIN_FRAC of each product's K slices, parks its fp32
  // partial sums in the workspace (partial set pbase + part), counts itself on counter set
  // `slot`, and the last piece to finish sums all pieces in part order and writes the item's
  // outputs.  nparts = 1: a whole item (f0 = 0, f1 = WIN_FRAC).
  int part, nparts, slot;
  int f0, f1, pbase;
};
constexpr int WIN_FRAC = 1 << 16;

// K slices [kb0, kb0 + nkb) of a CTA-pair rank-window item: its share of the whole K range of the
// product (d_in for the shrink, the covered d_out slices for dH).  The pieces of one item take
// consecutive shares, so their slice ranges tile the product's range exactly once.
__host__ __device__ __forceinline__ void win_krange(const WinItem& w, bool dh, int kmain, int& kb0, int& nkb) {
  const int b = dh ? w.dh_kb0 : 0, n = dh ? w.dh_nkb : kmain;
  const int lo = static_cast<int>(static_cast<long long>(n) * w.f0 / WIN_FRAC);
  const int hi = static_cast<int>(static_cast<long long>(n) * w.f1 / WIN_FRAC);
  kb0 = b + lo;
  nkb = hi - lo;
}

// Weight-gradient work item (dA / dB): one 256-row block of d_in (dA) or d_out (dB), one
// job, its 64-token half-tiles [ga, gb), chunks [q0, q0 + nq) of its rank window (nq <= MAX_ITEM_CHUNKS).
// An item whose tokens the schedule cuts across CTAs runs as `nparts` parts (token ranges in
// order, `part` = this one's index): each part parks its fp32 sums in the workspace (nq units of
// WG_UNIT floats from unit pbase + part * nq) and counts itself on counter set `cnt`; the last part
// to arrive adds the parts in part order and writes the gradient.  nparts = 1: a whole item.
struct WItem {
  int row0, seg, ga, gb, q0, nq;
  int part, nparts, pbase, cnt;
  int c0, r;    // the job's window start and rank, and its gradient (dAt for dA, dBt for dB; null in
  float* out;   // a shared-input pack, whose adapters the epilogue reads from the adapter table)
};
constexpr int WG_UNIT = 2 * BM * CHUNK_COLS;   // floats of one part's sums per chunk (256 rows x 64 columns)

struct AdamItem {
  float* p;
  const float* g;
  float* m;
  float* v;
  int count;
  // the bf16 shadow this piece's new values are copied to (when the step refreshes the shadows):
  // 1 = At_all, contiguous from element sh_base; 2 = Bt_all, element e of the tensor at
  // sh_base + (e / sh_r) * C + e % sh_r, the piece starting at tensor element sh_e0
  int sh_kind;
  long long sh_base;
  int sh_r;
  int sh_e0;
  long long pad0;
};

struct GemmArgs {
  int N;               // tokens
  int d_in, d_out;
  int kmain;           // 64-wide K slices of the main product (FWD/BWD/SHRINK/DH)
  int n_items;
  int n_tiles_n;       // FWD/BWD: output column tiles of 256
  int n_full_items;    // CTA-pair base GEMMs: items from here on are half-width tiles (see gemm_2sm.cu)
  int group_m;         // FWD/BWD raster: tiles per group (token tiles, or output tiles if raster_n)
  int raster_n;        // CTA-pair base GEMMs: 1 = groups of output tiles sweep the token pairs
  int n_mtiles;
  const MTile* mtiles;
  const WinItem* win;
  const WItem* witems;
  const DevSeg* segs;
  uint8_t* img_out;        // staged images written by the epilogue (SHRINK/DH)
  void* out;               // Y / dX (bf16)
  float* hout;             // H / dH (fp32)
  int ld_out;              // row stride (elements) of `out`
  int* err;                // device status word
  unsigned long long timeout_ns;
  int pdl;                 // launched with programmatic dependent launch
  int debug_drop;          // test hook: CTA 0 arms its first slot but issues no copy into it
  float* partials;         // fp32 partial sums of items split across CTAs (workspace)
  int* part_cnt;           // ... and their arrival counters (pair items: slot, CTA of the pair,
                           // row quarter; dA / dB items: counter set, row quarter, row half)
  const int* cta_first;    // dA / dB: CTA c runs items [cta_first[c], cta_first[c + 1]); CTA-pair shrink /
                           // dH: pair p runs [cta_first[p], cta_first[p + 1]) (null: round robin)
  // Shared-input packs (several adapters per job): per packed column, its adapter (-1 in the
  // padding) and scale.  Null for plans with one adapter per job, whose kernels read the job's.
  const DevSub* subs;      // job j's adapters are subs[j * n_groups .. j * n_groups + n_groups)
  const int* col_sub;
  const float* col_scale;
  int n_groups;
};

// Status codes written to the device status word (first one wins).
constexpr int DEV_ERR_TIMEOUT_PRODUCER = 0x101;
constexpr int DEV_ERR_TIMEOUT_MMA = 0x102;
constexpr int DEV_ERR_TIMEOUT_EPILOGUE = 0x103;
constexpr int DEV_ERR_TIMEOUT_TEARDOWN = 0x104;

// ---------------------------------------------------------------------------------------
// inline PTX wrappers
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after `timeout_ns` or when another
// role of the CTA has already given up (`abort_flag`).  On giving up it records `code` in the
// device status word (first error wins) and returns false; it never traps.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                          int code, unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}

// 2-D TMA tile load into shared memory, completing `bytes` on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 cache policy (see l2_policy_*).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 policies: data streamed once (evict first) and small operands re-read by many CTAs (evict last).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Contiguous bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Pull a 2-D box into L2 only (no shared-memory destination, no completion tracking).
__device__ __forceinline__ void prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: wait until the previous kernel in the stream has completed and
// its writes are visible (a no-op when the kernel was launched without the attribute), and let
// the next kernel start its prologue.  Every kernel calls griddep_wait() before its first global
// memory access, so overlapping launches never change results.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --- tcgen05 -----------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 consecutive fp32 columns of TMEM -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading/stride byte
// offsets, descriptor version 1, 128-byte swizzle.  For K-major operands the stride byte
// offset is the distance between 8-row atoms (1024 B) and the leading offset is unused; for
// MN-major operands the leading offset is the distance between 64-element MN blocks and the
// stride offset the distance between 8-deep K groups.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;   // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;   // SWIZZLE_128B
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                  // D format: fp32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)           // A major-ness
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// Byte offset of element (row, col) in a [rows x 64] bf16 tile stored as 128B-swizzled
// 8-row atoms (the layout TMA SWIZZLE_128B produces and the MMA descriptors expect).
__host__ __device__ __forceinline__ uint32_t swz128_offset(uint32_t row, uint32_t col) {
  const uint32_t chunk = (col >> 3) & 7u;
  return row * 128u + (((chunk ^ (row & 7u)) << 4) | ((col & 7u) << 1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Raise a kernel's dynamic shared-memory limit on the current device, once per device (the
// attribute is per device; `done` is the kernel's bitmask of devices already set).
template <typename K>
inline cudaError_t ensure_smem_attr(K kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launch `kernel` on `stream`, allowed to overlap the previous kernel's tail when `pdl`.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace mlora
