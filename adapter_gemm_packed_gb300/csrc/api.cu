// C ABI of the packed multi-adapter LoRA layer: planner, workspace layout, tensor maps and the
// launch sequences of forward / backward / AdamW.  See include/mlora.h for the contract.
//
// The planner is the host half of the rank-aware nano-batch scheduler ("tLoRA: Efficient
// Multi-LoRA Training with Elastic Shared Super-Models", abstract: rank-aware nano-batches;
// "PLoRA: Efficient Concurrent LoRA Training for Large Language Models", §9.2: tile along
// tokens / hidden dims, never along the rank).  It lays every job's rank window side by side in
// one packed rank space (windows padded to 16 columns, cut into 64-column chunks), maps each
// 128-token tile to the jobs and chunks it covers, and builds one static work list per kernel:
//   * base GEMMs: (256-token pair x 256 output columns) on CTA pairs, rastered in groups whose
//     resident panels fit the L2 (raster.cuh);
//   * shrink / dH: (token tile, <= 2 64-column chunks of its window), or on CTA pairs (256-token
//     pair, <= 4 chunks) laid out per pair and per product, the items past the even share cut
//     along K;
//   * dA / dB: (256-row block of d_in / d_out, job, <= 2 chunks) laid out per CTA, by greedy list
//     scheduling in job order or by McNaughton's wrap-around rule with items cut along their tokens.
#include <algorithm>
#include <array>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <limits>
#include <new>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "mlora.h"
#include "raster.cuh"
#include "pair.cuh"

namespace mlora {
template <int MODE>
cudaError_t launch_seg_gemm(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                            const GemmArgs&, int, cudaStream_t);
template <int MODE>
cudaError_t launch_gemm_2sm(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                            const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const GemmArgs&, int,
                            cudaStream_t);
template <int MODE>
cudaError_t launch_gemm_2sm_w4(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                               const CUtensorMap&, const GemmArgs&, int, cudaStream_t);
template <int MODE>
cudaError_t launch_win_2sm(const CUtensorMap&, const CUtensorMap&, const GemmArgs&, int, cudaStream_t);
cudaError_t launch_pack_fwd(const DevSub*, const int*, int, int, int, __nv_bfloat16*, __nv_bfloat16*, int,
                            cudaStream_t, bool);
cudaError_t launch_h_images(const DevSeg*, const float*, const MTile*, const int*, int, long long, const float*,
                            uint8_t*, cudaStream_t, bool);
cudaError_t launch_adamw(const AdamItem*, int, float, float, float, float, float, int, int, cudaStream_t, bool,
                         __nv_bfloat16*, __nv_bfloat16*, int);
cudaError_t launch_w4_expand(const void*, const float*, __nv_bfloat16*, int, int, int, cudaStream_t, bool);
cudaError_t launch_f32_forward(const DevSeg*, int, long long, int, int, long long, int, int, int, const float*,
                               const float*, float*, float*, cudaStream_t);
cudaError_t launch_f32_backward(const DevSeg*, int, long long, int, int, long long, int, int, int, const float*,
                                const float*, const float*, const float*, float*, float*, cudaStream_t);
}  // namespace mlora

using namespace mlora;

namespace {

thread_local std::string g_last_error;

}  // namespace

namespace mlora {
// Lets other translation units of the library report a message through mlora_last_error().
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace mlora

namespace {

mlora_status fail(mlora_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

mlora_status cuda_fail(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return MLORA_ERR_CUDA;
}

constexpr int ADAM_CHUNK = 4096;
constexpr int MAX_RANK = 256;
constexpr unsigned long long DEFAULT_TIMEOUT_NS = 4000000000ull;   // 4 s
constexpr unsigned long long SHORT_TIMEOUT_NS = 1000000ull;        // 1 ms

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over a row-major [outer, inner] matrix with a (box_inner x box_outer) box,
// 128-byte swizzle, zero fill outside the matrix.
mlora_status make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_elems,
                      uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return fail(MLORA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_elems * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] box %ux%u", static_cast<int>(r),
             static_cast<unsigned long long>(outer), static_cast<unsigned long long>(inner), box_inner, box_outer);
    return fail(MLORA_ERR_CUDA, buf);
  }
  return MLORA_OK;
}

// 2-D map without swizzle (4-bit codes as bytes, fp32 scales).
mlora_status make_map_plain(CUtensorMap* map, CUtensorMapDataType dt, uint32_t esize, const void* base, uint64_t inner,
                            uint64_t outer, uint64_t row_elems, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return fail(MLORA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_elems * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLORA_ERR_CUDA, "cuTensorMapEncodeTiled failed for a 4-bit weight map");
  return MLORA_OK;
}

}  // namespace

struct mlora_plan_s {
  mlora_problem prob{};
  int n_segs = 0;                       // user entries: n_jobs x n_groups, job-major
  int n_jobs = 0, n_groups = 1;
  bool grouped = false;                 // more than one output-column group (shared-input pack)
  std::vector<mlora_group> groups;
  std::vector<mlora_segment> user;
  std::vector<DevSeg> segs;             // one per job
  std::vector<DevSub> subs;             // one per user entry
  std::vector<float> col_scale;         // per packed column (chunk-padded), 0 in padding
  int C_total = 0, n_chunks = 0, n_mtiles = 0, max_rank = 0, max_tokens = 0;
  long long n_images = 0, h_elems = 0;
  std::vector<MTile> mtiles;
  std::vector<int> img_tile;
  std::vector<int> col_sub;             // per packed column (chunk-padded), -1 in padding
  std::vector<WinItem> win;             // shrink / dH items of the single-CTA engine (tile, <= 2 chunks)
  std::vector<WinItem> win2;            // the shrink on CTA pairs (tile = pair, 2 or 4 chunks), per-pair lists
  bool win_pairs = false;               // which of the two the shrink / dH launches run
  std::vector<int> win2_first;          // shrink: pair p runs win2[win2_first[p] .. win2_first[p + 1])
  std::vector<WinItem> win2d;           // dH on CTA pairs: the same items laid out for dH's K range
  std::vector<int> win2d_first;
  int n_split = 0, win_units = 0;       // pair items cut along K (see build_tables), and their pieces
                                        // (the larger of the two products')
  std::vector<WItem> da, db;             // dA / dB items, CTA by CTA (see build_tables)
  std::vector<int> da_first, db_first;   // CTA c runs items [first[c], first[c + 1])
  int da_sets = 0, db_sets = 0;          // items cut across CTAs (one arrival-counter set each)
  int da_units = 0, db_units = 0;        // their parked partial sums, in units of WG_UNIT floats
  std::vector<AdamItem> adam;
  bool can_backward = false, can_adamw = false;
  size_t off_shadow = 0, off_partials = 0, off_himg = 0, off_dhimg = 0, off_wexp = 0, ws_bytes = 0;
  bool w4_fused = false;   // 4-bit base expanded inside the GEMMs instead of into the workspace
  int group_m = 8;
  // device
  bool on_device = false;
  int device = 0, num_sms = 148;
  void* dev_block = nullptr;
  DevSeg* d_segs = nullptr;
  MTile* d_mtiles = nullptr;
  int* d_img_tile = nullptr;
  DevSub* d_subs = nullptr;
  int* d_col_sub = nullptr;
  float* d_col_scale = nullptr;
  WinItem* d_win = nullptr;
  WinItem* d_win2 = nullptr;
  WItem* d_da = nullptr;
  WItem* d_db = nullptr;
  int* d_da_first = nullptr;
  int* d_db_first = nullptr;
  int* d_win2_first = nullptr;
  WinItem* d_win2d = nullptr;
  int* d_win2d_first = nullptr;
  AdamItem* d_adam = nullptr;
  int* d_err = nullptr;
  int* d_part_cnt = nullptr;            // arrival counters of the split items: pair items, then dA's,
                                        // then dB's (zeroed at upload)
  unsigned long long timeout_ns = DEFAULT_TIMEOUT_NS;
  bool pdl = true;
  bool debug_drop = false;             // single-CTA shrink withholds one copy (test hook)
  bool debug_drop_pairs = false;       // the forward's CTA-pair kernels withhold one copy (test hook)
  // what the last forward left in a workspace (used with MLORA_REUSE_STAGING)
  bool reuse_staging = false;
  bool staged_valid = false;
  const void* staged_ws = nullptr;
  const float* staged_H = nullptr;
  bool shadows_valid = false;          // the bf16 shadows in shadows_ws match the fp32 masters
  const void* shadows_ws = nullptr;
  const void* staged_wq = nullptr;     // 4-bit base whose bf16 expansion the workspace holds
  const float* staged_wscale = nullptr;
  // optional per-kernel timing with CUDA events recorded on the launching stream
  bool profiling = false;
  std::vector<cudaEvent_t> ev_pool;
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> ev_pending;
  size_t ev_next = 0;
};

namespace mlora {
// Forget whatever the plan recorded about `workspace` (shadows, staged images, 4-bit
// expansion), so that its next forward or backward with that buffer rebuilds them.  For
// scratch that other plans also write, which the plan's own bookkeeping cannot see.
void forget_workspace(const mlora_plan_t* Pc, const void* workspace) {
  mlora_plan_t* P = const_cast<mlora_plan_t*>(Pc);
  if (P->shadows_ws == workspace) {
    P->shadows_valid = false;
    P->shadows_ws = nullptr;
  }
  if (P->staged_ws == workspace) {
    P->staged_valid = false;
    P->staged_ws = nullptr;
    P->staged_H = nullptr;
    P->staged_wq = nullptr;
    P->staged_wscale = nullptr;
  }
}

bool plan_is_w4(const mlora_plan_t* P) { return P->prob.dtype == MLORA_BF16_W4; }
}  // namespace mlora

namespace {

mlora_status validate(const mlora_problem* p, const mlora_group* groups, int32_t n_groups, const mlora_segment* s,
                      int32_t n) {
  if (!p || !s || !groups) return fail(MLORA_ERR_INVALID, "null problem, group or segment table");
  if (n_groups < 1) return fail(MLORA_ERR_INVALID, "n_groups must be >= 1");
  if (n < 1) return fail(MLORA_ERR_INVALID, "n_segs must be >= 1");
  if (n % n_groups) return fail(MLORA_ERR_INVALID, "n_segs must be a multiple of n_groups (one entry per job and group)");
  if (p->dtype != MLORA_F32 && p->dtype != MLORA_BF16 && p->dtype != MLORA_BF16_W4)
    return fail(MLORA_ERR_INVALID, "unknown dtype");
  if (p->dtype == MLORA_BF16_W4 && p->d_in % 64)
    return fail(MLORA_ERR_UNSUPPORTED, "a 4-bit base needs d_in a multiple of 64");
  if (p->dtype == MLORA_BF16_W4 && (p->flags & MLORA_W4_FUSED) && (p->flags & MLORA_GEMM_SINGLE_CTA))
    return fail(MLORA_ERR_UNSUPPORTED, "the fused 4-bit GEMMs run on CTA pairs only");
  if (p->d_in < 1 || p->d_out < 1) return fail(MLORA_ERR_INVALID, "d_in and d_out must be >= 1");
  const int q = p->dtype == MLORA_F32 ? 4 : 8;
  if (p->d_in % q || p->d_out % q)
    return fail(MLORA_ERR_UNSUPPORTED, "d_in and d_out must be multiples of 8 (bf16) or 4 (fp32)");
  if (p->n_tokens < 1 || p->n_tokens > 0x7fffffffLL) return fail(MLORA_ERR_INVALID, "n_tokens out of range");
  if (n_groups > 1 && p->dtype == MLORA_F32)
    return fail(MLORA_ERR_UNSUPPORTED, "shared-input packs (several groups) need a bf16 plan");
  {
    long long o = 0;
    for (int g = 0; g < n_groups; ++g) {
      if (groups[g].col_offset != o || groups[g].d_out < 1)
        return fail(MLORA_ERR_INVALID, "groups must tile [0, d_out) in order, each at least one column wide");
      o += groups[g].d_out;
    }
    if (o != p->d_out) return fail(MLORA_ERR_INVALID, "the groups' widths must add up to d_out");
  }
  long long expect = 0;
  for (int i = 0; i < n; ++i) {
    const mlora_segment& g = s[i];
    const mlora_segment& first = s[i - i % n_groups];   // the job's entry for group 0
    char buf[160];
    if (i % n_groups == 0) {
      if (g.tok_offset != expect) {
        snprintf(buf, sizeof buf, "segment %d starts at row %lld, expected %lld (segments must tile [0, N) in order)", i,
                 static_cast<long long>(g.tok_offset), expect);
        return fail(MLORA_ERR_INVALID, buf);
      }
    } else if (g.tok_offset != first.tok_offset || g.n_tokens != first.n_tokens) {
      snprintf(buf, sizeof buf, "segment %d: a job's entries for every group must cover the same rows", i);
      return fail(MLORA_ERR_INVALID, buf);
    }
    if (g.n_tokens < 1) {
      snprintf(buf, sizeof buf, "segment %d has n_tokens < 1", i);
      return fail(MLORA_ERR_INVALID, buf);
    }
    if (g.rank < 1) {
      snprintf(buf, sizeof buf, "segment %d has rank < 1", i);
      return fail(MLORA_ERR_INVALID, buf);
    }
    if (g.rank > MAX_RANK) {
      snprintf(buf, sizeof buf, "segment %d has rank %d > %d", i, g.rank, MAX_RANK);
      return fail(MLORA_ERR_UNSUPPORTED, buf);
    }
    if (!std::isfinite(g.scale)) {
      snprintf(buf, sizeof buf, "segment %d has a non-finite scale", i);
      return fail(MLORA_ERR_INVALID, buf);
    }
    if (!g.At || !g.Bt) {
      snprintf(buf, sizeof buf, "segment %d: At and Bt are required", i);
      return fail(MLORA_ERR_INVALID, buf);
    }
    const float* ptrs[8] = {g.At, g.Bt, g.dAt, g.dBt, g.mA, g.vA, g.mB, g.vB};
    for (const float* ptr : ptrs)
      if (ptr && !aligned16(ptr)) {
        snprintf(buf, sizeof buf, "segment %d: adapter buffers must be 16-byte aligned", i);
        return fail(MLORA_ERR_INVALID, buf);
      }
    if (i % n_groups == n_groups - 1) expect += g.n_tokens;
  }
  if (expect != p->n_tokens) {
    char buf[160];
    snprintf(buf, sizeof buf, "segments cover %lld rows but n_tokens is %lld", expect,
             static_cast<long long>(p->n_tokens));
    return fail(MLORA_ERR_INVALID, buf);
  }
  return MLORA_OK;
}

void build_tables(mlora_plan_t* P) {
  const mlora_problem& pr = P->prob;
  const long long N = pr.n_tokens;
  const int G = P->n_groups;
  // Jobs and the packed rank space.  Job j's adapters (one per group) sit side by side in its
  // window in group order, without padding between them; the window is padded to RANK_PAD.
  int c = 0;
  long long h = 0;
  P->segs.resize(P->n_jobs);
  P->subs.resize(P->n_segs);
  P->can_backward = P->can_adamw = true;
  for (int j = 0; j < P->n_jobs; ++j) {
    const mlora_segment& u0 = P->user[static_cast<size_t>(j) * G];
    DevSeg& d = P->segs[j];
    d.off = u0.tok_offset;
    d.n = u0.n_tokens;
    d.c = c;
    d.pad0 = 0;
    d.h_off = h;
    int R = 0;
    for (int g = 0; g < G; ++g) {
      const int i = j * G + g;
      const mlora_segment& u = P->user[i];
      DevSub& sb = P->subs[i];
      sb.At = u.At;
      sb.Bt = u.Bt;
      sb.dAt = u.dAt;
      sb.dBt = u.dBt;
      sb.c0 = c + R;
      sb.r = u.rank;
      sb.o_lo = P->groups[g].col_offset;
      sb.o_hi = P->groups[g].col_offset + P->groups[g].d_out;
      sb.s = u.scale;
      sb.job = j;
      sb.pad0 = sb.pad1 = 0;
      R += u.rank;
      P->max_rank = std::max(P->max_rank, u.rank);
      P->max_tokens = std::max(P->max_tokens, u.n_tokens);
      if (!u.dAt || !u.dBt) P->can_backward = false;
      if (!u.dAt || !u.dBt || !u.mA || !u.vA || !u.mB || !u.vB) P->can_adamw = false;
    }
    // one adapter per job: the job carries it (the kernels' fast paths read these)
    d.r = R;
    d.rp = static_cast<int>(round_up(R, RANK_PAD));
    d.s = G == 1 ? u0.scale : 0.f;
    d.At = G == 1 ? u0.At : nullptr;
    d.Bt = G == 1 ? u0.Bt : nullptr;
    d.dAt = G == 1 ? u0.dAt : nullptr;
    d.dBt = G == 1 ? u0.dBt : nullptr;
    c += d.rp;
    h += static_cast<long long>(d.n) * R;
  }
  P->C_total = c;
  P->h_elems = h;
  P->n_chunks = (c + CHUNK_COLS - 1) / CHUNK_COLS;
  P->col_sub.assign(static_cast<size_t>(P->n_chunks) * CHUNK_COLS, -1);
  P->col_scale.assign(static_cast<size_t>(P->n_chunks) * CHUNK_COLS, 0.f);
  for (int i = 0; i < P->n_segs; ++i)
    for (int t = 0; t < P->subs[i].r; ++t) {
      P->col_sub[P->subs[i].c0 + t] = i;
      P->col_scale[P->subs[i].c0 + t] = P->subs[i].s;
    }

  // token tiles -> jobs -> chunks -> staged images
  P->n_mtiles = static_cast<int>((N + BM - 1) / BM);
  P->mtiles.resize(P->n_mtiles);
  int j = 0;
  long long img = 0;
  for (int t = 0; t < P->n_mtiles; ++t) {
    const long long r0 = static_cast<long long>(t) * BM, r1 = std::min(N, r0 + BM) - 1;
    while (P->segs[j].off + P->segs[j].n <= r0) ++j;
    int k = j;
    while (P->segs[k].off + P->segs[k].n <= r1) ++k;
    MTile& m = P->mtiles[t];
    m.seg_first = j;
    m.seg_last = k;
    const int c_lo = P->segs[j].c, c_hi = P->segs[k].c + P->segs[k].rp;
    m.q_lo = c_lo / CHUNK_COLS;
    m.nch = (c_hi + CHUNK_COLS - 1) / CHUNK_COLS - m.q_lo;
    m.img_off = static_cast<int>(img);
    m.pad0 = m.pad1 = m.pad2 = 0;
    img += m.nch;
  }
  // The 2-CTA base GEMMs run 256-token tiles whose rank-term K extension is one MMA over both
  // 128-token halves, so both halves of a pair stage the union of their chunk ranges.
  img = 0;
  for (int t = 0; t < P->n_mtiles; t += 2) {
    MTile& a = P->mtiles[t];
    if (t + 1 < P->n_mtiles) {
      MTile& b = P->mtiles[t + 1];
      const int lo = std::min(a.q_lo, b.q_lo), hi = std::max(a.q_lo + a.nch, b.q_lo + b.nch);
      a.q_lo = b.q_lo = lo;
      a.nch = b.nch = hi - lo;
    }
    for (int u = t; u < std::min(t + 2, P->n_mtiles); ++u) {
      P->mtiles[u].img_off = static_cast<int>(img);
      img += P->mtiles[u].nch;
    }
  }
  P->n_images = img;
  P->img_tile.resize(img);
  for (int t = 0; t < P->n_mtiles; ++t)
    for (int e = 0; e < P->mtiles[t].nch; ++e) P->img_tile[P->mtiles[t].img_off + e] = t;

  // dH reads only the d_out slices that the adapters owning the item's columns cover
  auto dh_range = [&](WinItem& w, int q0, int nq) {
    int o_lo = pr.d_out, o_hi = 0;
    for (int c = q0 * CHUNK_COLS; c < std::min(P->C_total, (q0 + nq) * CHUNK_COLS); ++c) {
      const int a = P->col_sub[c];
      if (a < 0) continue;
      o_lo = std::min(o_lo, P->subs[a].o_lo);
      o_hi = std::max(o_hi, P->subs[a].o_hi);
    }
    if (o_hi <= o_lo) o_lo = 0, o_hi = std::min(pr.d_out, BK);
    w.dh_kb0 = o_lo / BK;
    w.dh_nkb = (o_hi + BK - 1) / BK - w.dh_kb0;
  };
  // shrink / dH work, single-CTA engine: one item per (tile, <= MAX_ITEM_CHUNKS chunks)
  P->win.clear();
  long long chunk_sum = 0;
  for (int t = 0; t < P->n_mtiles; ++t) {
    const MTile& m = P->mtiles[t];
    chunk_sum += m.nch;
    for (int q = 0; q < m.nch; q += MAX_ITEM_CHUNKS) {
      WinItem w{};
      w.tile = t;
      w.q0 = m.q_lo + q;
      w.nq = std::min(MAX_ITEM_CHUNKS, m.nch - q);
      w.nparts = 1;
      w.f1 = WIN_FRAC;
      dh_range(w, w.q0, w.nq);
      P->win.push_back(w);
    }
  }
  // ... and on CTA pairs: one item per (256-token pair, <= 4 chunks of its shared window), the
  // chunk count rounded up to even so that each CTA holds whole chunks
  P->win2.clear();
  for (int t = 0; t < P->n_mtiles; t += 2) {
    const MTile& m = P->mtiles[t];
    for (int q = 0; q < m.nch; q += 4) {
      WinItem w{};
      w.tile = t / 2;
      w.q0 = m.q_lo + q;
      const int real = std::min(4, m.nch - q);
      w.nq = real + (real & 1);
      w.nparts = 1;
      w.f1 = WIN_FRAC;
      dh_range(w, w.q0, real);
      P->win2.push_back(w);
    }
  }
  // Pairs halve the rank operand's bytes per token and the re-reads of X / dY for wide windows;
  // a one-chunk window gains nothing (it is padded to two), so pairs run when tiles average
  // more than 1.25 chunks, unless a flag forces either engine.
  P->win_pairs = 4 * chunk_sum > 5LL * P->n_mtiles;
  if (pr.flags & MLORA_WINDOW_PAIRS) P->win_pairs = true;
  if (pr.flags & MLORA_WINDOW_SINGLE) P->win_pairs = false;
  if (P->debug_drop) P->win_pairs = false;   // the copy-withholding hook lives in the single-CTA shrink

  // CTA-pair schedules of the shrink and of dH: for each product a list per pair.  The modelled
  // cost of an item, in KB per CTA, is what it streams (per 64-wide K slice of the product, 16 KB
  // of X or dY and 8 KB per rank-operand chunk the CTA holds), its images (16 KB per chunk) and a
  // start-up.  First the items go whole, in tile order, each to the least-loaded pair, while that
  // pair then stays within an eighth of the item above the average load: the first waves run like
  // a round robin (a tile's items, which read the same X / dY rows, side by side).  The rest are
  // laid out by McNaughton's wrap-around rule over the pairs in ascending order of load: each pair
  // is filled up to a level T, the item at its end is cut there along K (at least 16 K slices per
  // piece) and its rest starts the next pair; T is the level whose layout has the smallest largest
  // load (scanned below).  A cut piece also parks its fp32 sums and the item's
  // last piece reads all of them back: 64 KB per chunk per piece in the model.  Against a round
  // robin this fills the last wave's idle pairs (one item of a wave's time left to a few pairs)
  // and the pairs a pack with fewer items than pairs leaves idle.  The two products' K ranges
  // differ (d_in against the d_out slices dH covers), so each gets its own layout; the launches
  // run one after the other and share the partial sums and counters.
  auto pair_schedule = [&](const std::vector<WinItem>& v, bool dh, std::vector<WinItem>& out,
                           std::vector<int>& first, int& sets, int& units) {
    out.clear();
    first.clear();
    sets = units = 0;
    const int NP = std::max(1, P->num_sms / 2);
    const int kin = (pr.d_in + BK - 1) / BK;
    auto ks = [&](const WinItem& w) { return dh ? w.dh_nkb : kin; };
    auto var = [&](const WinItem& w) { return ks(w) * (16.0 + 8.0 * (w.nq / 2)); };
    auto fix = [&](const WinItem& w) { return 32.0 + 16.0 * w.nq; };
    auto cutc = [&](const WinItem& w) { return 64.0 * w.nq; };
    // the smallest share of a piece: 16 K slices (an item shorter than 32 slices is never cut)
    auto fmin = [&](const WinItem& w) {
      const int mk = std::max(1, ks(w));
      return static_cast<int>((16LL * WIN_FRAC + mk - 1) / mk);
    };
    std::vector<std::vector<WinItem>> lists(NP);
    std::vector<double> load(NP, 0.0);
    size_t i = 0;
    if (P->win_pairs) {
      double total = 0;
      for (const WinItem& w : v) total += var(w) + fix(w);
      const double avg = total / NP;
      for (; i < v.size(); ++i) {
        int p = 0;   // the least-loaded pair (lowest index among equals)
        for (int k = 1; k < NP; ++k)
          if (load[k] < load[p]) p = k;
        const double c = var(v[i]) + fix(v[i]);
        if (load[p] + c > avg + c / 8) break;
        lists[p].push_back(v[i]);
        load[p] += c;
      }
    } else {
      for (; i < v.size(); ++i) lists[i % NP].push_back(v[i]);   // not launched: whole items
    }
    if (i < v.size()) {
      std::vector<int> order(NP);
      for (int k = 0; k < NP; ++k) order[k] = k;
      std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return load[x] < load[y]; });
      std::vector<std::vector<WinItem>> add;
      // lays out items i.. at level T (the last pair in the order takes whatever is left, if the
      // layout reaches it); returns the largest load and leaves the per-pair pieces in `add`
      auto lay_out = [&](double T) {
        add.assign(NP, {});
        std::vector<double> ld = load;
        sets = units = 0;
        int oi = 0;
        for (size_t k = i; k < v.size(); ++k) {
          const WinItem& w = v[k];
          const int fm = fmin(w);
          std::vector<std::array<int, 3>> pieces;   // (pair, f0, f1)
          int f = 0;
          while (f < WIN_FRAC) {
            const int p = order[oi];
            const int rest = WIN_FRAC - f;
            int take;
            if (oi == NP - 1) {
              take = rest;   // the last pair takes whatever is left
            } else {
              const double room = T - ld[p] - fix(w) - cutc(w);
              take = room <= 0 ? 0 : static_cast<int>(std::min<double>(rest, std::floor(room / var(w) * WIN_FRAC)));
              if (take < rest) {
                if (take < fm) {
                  // a piece of the smallest share here overfills this pair, none leaves its room
                  // empty: take the smaller of the two deviations (an empty pair always takes one)
                  const bool empty = lists[p].empty() && add[p].empty();
                  if (!empty && room < 0.5 * fm / WIN_FRAC * var(w)) {
                    ++oi;
                    continue;
                  }
                  take = std::min(rest, fm);
                }
                const int r2 = rest - take;
                if (r2 > 0 && r2 < fm)   // no stub: take it all, or leave the smallest share
                  take = (2 * r2 < fm || rest < 2 * fm) ? rest : rest - fm;
              }
            }
            pieces.push_back({p, f, f + take});
            ld[p] += fix(w) + var(w) * take / WIN_FRAC + (take == WIN_FRAC ? 0.0 : cutc(w));
            add[p].push_back(w);   // filled in below
            f += take;
            if (f < WIN_FRAC) ++oi;
          }
          const int S = static_cast<int>(pieces.size());
          for (int q = 0; q < S; ++q) {
            WinItem& x = add[pieces[q][0]].back();
            x.part = q;
            x.nparts = S;
            x.f0 = pieces[q][1];
            x.f1 = pieces[q][2];
            x.slot = S > 1 ? sets : 0;
            x.pbase = S > 1 ? units : 0;
          }
          if (S > 1) {
            ++sets;
            units += S;
          }
        }
        return *std::max_element(ld.begin(), ld.end());
      };
      // The level: pieces of at least 16 slices make the largest load jump with T (a piece that
      // would fit only in part overfills a pair, or moves on and leaves its room empty), so T is
      // scanned from the average load up to 1.5x (and a few larger values) in steps of 0.2 %, and
      // the layout with the smallest largest load is kept (the lowest T among equals).
      double avg = 0;
      for (size_t k = i; k < v.size(); ++k) avg += var(v[k]) + fix(v[k]);
      for (int k = 0; k < NP; ++k) avg += load[k];
      avg /= NP;
      double best_T = avg, best = std::numeric_limits<double>::infinity();
      for (int step = 0; step <= 253; ++step) {
        const double T = avg * (step <= 250 ? 1.0 + 0.002 * step : 1.0 + (step - 249));
        const double span = lay_out(T);
        if (span < best) {
          best = span;
          best_T = T;
        }
      }
      lay_out(best_T);
      for (int k = 0; k < NP; ++k) lists[k].insert(lists[k].end(), add[k].begin(), add[k].end());
    }
    int used = NP;
    while (used > 1 && lists[used - 1].empty()) --used;
    for (int k = 0; k < used; ++k) {
      first.push_back(static_cast<int>(out.size()));
      out.insert(out.end(), lists[k].begin(), lists[k].end());
    }
    first.push_back(static_cast<int>(out.size()));
  };
  {
    const std::vector<WinItem> v = std::move(P->win2);
    int s_sets, s_units, d_sets, d_units;
    pair_schedule(v, false, P->win2, P->win2_first, s_sets, s_units);
    pair_schedule(v, true, P->win2d, P->win2d_first, d_sets, d_units);
    P->n_split = std::max(s_sets, d_sets);
    P->win_units = std::max(s_units, d_units);
  }

  // dA / dB work: (256-row block, job, <= MAX_ITEM_CHUNKS chunks) over the job's tokens.  A dB
  // block needs only the columns of the job's adapters whose output range meets it.  Items that
  // run at the same time should read the same X / dY rows (the neighbouring 256-column blocks of
  // one job's tokens): those reads then cover whole rows of the row-major tensor instead of
  // scattered 512-byte pieces (a schedule that ran one job's blocks one after the other on the
  // same CTA measured 1.3-1.5x slower).  Two schedules are built; the cut one is kept only where
  // its modelled end is far sooner:
  //  - greedy list scheduling of the items in job order (longest jobs first, then block, then
  //    chunks), each to the CTA with the least modelled load: consecutive items (one job's
  //    blocks) start at about the same time on different CTAs, and longest-first keeps the ends
  //    even when the items are small against a CTA's share T of the total.
  //  - McNaughton's wrap-around rule over the items in block order (then job = token order, then
  //    chunks), for few blocks and long jobs: each CTA takes its even share of the work still
  //    unassigned (T at first), the item at its end is cut there along its tokens (at a 64-token
  //    half-tile) and its rest starts the next CTA, so every CTA ends near T whatever the mix of
  //    job lengths.  The CTAs of
  //    the blocks' runs start at the same token offsets when the block count divides the CTA
  //    count (else at a few different offsets), so CTAs of different blocks still read the same
  //    rows together.  Pieces shorter than MIN_PART_HT half-tiles are not made.  A cut item's
  //    parts run first on their CTAs; the last one to finish sums all parts.
  constexpr int MIN_PART_HT = 4;
  auto wgrad = [&](int rows, bool by_output, std::vector<WItem>& items, std::vector<int>& first, int& sets,
                   int& units) {
    // modelled cost, in KB moved: per half-tile the streamed operand (32 KB) and the images (8 KB
    // per chunk); per piece its output (the gradient's 256 rows x 4 bytes, 1 KB, per column of the
    // job inside the item's chunks) and a start-up
    auto per_ht = [](int nq) { return 32.0 + 8.0 * nq; };
    auto fixed = [&](const WItem& w) {
      const DevSeg& d = P->segs[w.seg];
      const int lo = std::max(d.c, w.q0 * CHUNK_COLS), hi = std::min(d.c + d.r, (w.q0 + w.nq) * CHUNK_COLS);
      return 32.0 + std::max(0, hi - lo);
    };
    auto cost = [&](const WItem& w) { return fixed(w) + per_ht(w.nq) * (w.gb - w.ga); };
    // items of job i in row block r0
    auto block_items = [&](int i, int r0, std::vector<WItem>& out) {
      const DevSeg& d = P->segs[i];
      const int ga = static_cast<int>(d.off / 64);
      const int gb = static_cast<int>((d.off + d.n + 63) / 64);
      int c_lo = d.c + d.r, c_hi = d.c;
      for (int g = 0; g < G; ++g) {
        const DevSub& sb = P->subs[static_cast<size_t>(i) * G + g];
        if (by_output && (sb.o_hi <= r0 || sb.o_lo >= r0 + 2 * BM)) continue;
        c_lo = std::min(c_lo, sb.c0);
        c_hi = std::max(c_hi, sb.c0 + sb.r);
      }
      if (c_hi <= c_lo) return;
      const int qa = c_lo / CHUNK_COLS, qb = (c_hi + CHUNK_COLS - 1) / CHUNK_COLS;
      for (int q = qa; q < qb; q += MAX_ITEM_CHUNKS)
        out.push_back(WItem{r0, i, ga, gb, q, std::min(MAX_ITEM_CHUNKS, qb - q), 0, 1, 0, 0, d.c, d.r,
                            by_output ? d.dBt : d.dAt});
    };
    std::vector<WItem> v;   // block order
    for (int r0 = 0; r0 < rows; r0 += 2 * BM)
      for (int i = 0; i < P->n_jobs; ++i) block_items(i, r0, v);
    double total = 0;
    for (const WItem& w : v) total += cost(w);
    const int n_cta = std::max(1, P->num_sms);

    // greedy list scheduling in job order, longest jobs first
    std::vector<std::vector<WItem>> g_whole(n_cta);
    double g_span = 0;
    {
      std::vector<int> jobs(P->n_jobs);
      for (int i = 0; i < P->n_jobs; ++i) jobs[i] = i;
      std::stable_sort(jobs.begin(), jobs.end(), [&](int a, int b) { return P->segs[a].n > P->segs[b].n; });
      std::vector<WItem> u;
      for (int i : jobs)
        for (int r0 = 0; r0 < rows; r0 += 2 * BM) block_items(i, r0, u);
      std::vector<double> load(n_cta, 0.0);
      for (const WItem& w : u) {
        int lowest = 0;   // the least-loaded CTA (lowest index among equals)
        for (int k = 1; k < n_cta; ++k)
          if (load[k] < load[lowest]) lowest = k;
        g_whole[lowest].push_back(w);
        load[lowest] += cost(w);
      }
      g_span = *std::max_element(load.begin(), load.end());
    }

    // McNaughton over the block order.  A piece of a cut item also writes its partial sums (all
    // 64 columns of a chunk) and the item's last part reads them all back: 128 KB per chunk per
    // piece on top of its cost.  Each CTA takes up to T; T is the smallest budget (to 0.1 %, by
    // bisection) at which the last CTA's share stays within it as well.
    std::vector<std::vector<WItem>> m_cut, m_whole;
    double m_span = 0;
    int m_sets = 0, m_units = 0;
    {
      auto piece_cost = [&](const WItem& w, int nh, bool is_cut) {
        return fixed(w) + per_ht(w.nq) * nh + (is_cut ? 128.0 * w.nq : 0.0);
      };
      // lays the items out with budget T; returns the load of the last CTA (which takes whatever
      // is left) and sets m_span to the largest load
      auto lay_out = [&](double T) {
        m_cut.assign(n_cta, {});
        m_whole.assign(n_cta, {});
        std::vector<double> load(n_cta, 0.0);
        int c = 0;
        m_sets = 0;
        m_units = 0;
        for (const WItem& w : v) {
          std::vector<std::array<int, 3>> pieces;   // (CTA, first half-tile, end half-tile)
          int a = w.ga;
          while (a < w.gb) {
            const int nh = w.gb - a;
            const double room = T - load[c] - piece_cost(w, 0, true);
            int take = static_cast<int>(std::floor(room / per_ht(w.nq)));
            if (c == n_cta - 1 || take >= nh) {
              take = nh;   // the rest fits (or the last CTA takes it)
            } else {
              if (take < MIN_PART_HT) {
                // a piece of MIN_PART_HT here overfills this CTA, none leaves its room empty: take
                // the smaller of the two deviations
                const bool empty = m_cut[c].empty() && m_whole[c].empty();
                if (!empty && room < 0.5 * MIN_PART_HT * per_ht(w.nq)) {
                  ++c;
                  continue;
                }
                take = std::min(nh, MIN_PART_HT);
              }
              const int rest = nh - take;
              if (rest > 0 && rest < MIN_PART_HT)   // no stub: take it all, or leave MIN_PART_HT
                take = (2 * rest < MIN_PART_HT || nh < 2 * MIN_PART_HT) ? nh : nh - MIN_PART_HT;
            }
            pieces.push_back({c, a, a + take});
            (take == w.gb - w.ga ? m_whole : m_cut)[c].push_back(w);   // filled in below
            load[c] += piece_cost(w, take, take != w.gb - w.ga);
            a += take;
            if (a < w.gb) ++c;
          }
          const int S = static_cast<int>(pieces.size());
          for (int k = 0; k < S; ++k) {
            WItem& x = (S > 1 ? m_cut : m_whole)[pieces[k][0]].back();
            x.ga = pieces[k][1];
            x.gb = pieces[k][2];
            x.part = k;
            x.nparts = S;
            x.pbase = S > 1 ? m_units : 0;
            x.cnt = S > 1 ? m_sets : 0;
          }
          if (S > 1) {
            m_units += S * w.nq;
            ++m_sets;
          }
        }
        m_span = *std::max_element(load.begin(), load.end());
        return load[n_cta - 1];
      };
      double lo = total / n_cta, hi = 1.25 * lo;
      while (lay_out(hi) > hi && hi < 64 * total) hi *= 1.25;
      while (hi - lo > 0.001 * hi) {
        const double mid = 0.5 * (lo + hi);
        (lay_out(mid) > mid ? lo : hi) = mid;
      }
      lay_out(hi);
    }
    // The cut schedule only where the greedy one is far off: its parts' partial sums and the last
    // part's sum cost more than the model counts (measured: the cut schedule lost at a modelled
    // 0.79 of the greedy end on a 16-block dA, and won at about 0.5 on a 4-block dB).
    const bool use_m = m_span < 0.7 * g_span;
    std::vector<std::vector<WItem>> cut, whole;
    if (use_m) {
      cut = std::move(m_cut);
      whole = std::move(m_whole);
      sets = m_sets;
      units = m_units;
    } else {
      cut.assign(n_cta, {});
      whole = std::move(g_whole);
      sets = 0;
      units = 0;
    }
    items.clear();
    first.clear();
    for (int k = 0; k < n_cta; ++k) {
      if (cut[k].empty() && whole[k].empty()) break;   // both schedules fill CTAs in index order
      first.push_back(static_cast<int>(items.size()));
      items.insert(items.end(), cut[k].begin(), cut[k].end());
      items.insert(items.end(), whole[k].begin(), whole[k].end());
    }
    first.push_back(static_cast<int>(items.size()));
  };
  wgrad(pr.d_in, false, P->da, P->da_first, P->da_sets, P->da_units);
  wgrad(pr.d_out, true, P->db, P->db_first, P->db_sets, P->db_units);

  // AdamW pieces
  P->adam.clear();
  if (P->can_adamw) {
    for (int i = 0; i < P->n_segs; ++i) {
      const mlora_segment& u = P->user[i];
      const DevSub& sb = P->subs[i];
      const long long width = sb.o_hi - sb.o_lo;
      // shadow copies: At rows are rows c0.. of At_all (contiguous); B^T row o, rank t is
      // Bt_all[o_lo + o][c0 + t]
      struct T { float *p, *g, *m, *v; long long n; int kind; long long base; } ts[2] = {
          {u.At, u.dAt, u.mA, u.vA, static_cast<long long>(u.rank) * pr.d_in, 1,
           static_cast<long long>(sb.c0) * pr.d_in},
          {u.Bt, u.dBt, u.mB, u.vB, static_cast<long long>(u.rank) * width, 2,
           static_cast<long long>(sb.o_lo) * P->C_total + sb.c0}};
      for (const T& tt : ts)
        for (long long s0 = 0; s0 < tt.n; s0 += ADAM_CHUNK) {
          AdamItem a{};
          a.p = tt.p + s0;
          a.g = tt.g + s0;
          a.m = tt.m + s0;
          a.v = tt.v + s0;
          a.count = static_cast<int>(std::min<long long>(ADAM_CHUNK, tt.n - s0));
          a.sh_kind = tt.kind;
          a.sh_base = tt.kind == 1 ? tt.base + s0 : tt.base;
          a.sh_r = u.rank;
          a.sh_e0 = static_cast<int>(s0);
          P->adam.push_back(a);
        }
    }
  }

  // workspace: the two bf16 shadows At_all, Bt_all (rebuilt by every forward and backward call),
  // then the two image sets
  if (pr.dtype != MLORA_F32) {
    const size_t shadow = round_up(static_cast<size_t>(P->C_total) * pr.d_in * 2, 1024) +
                          round_up(static_cast<size_t>(P->C_total) * pr.d_out * 2, 1024);
    P->off_shadow = 0;
    // fp32 partial sums of split items, one region shared by the launches that use it in turn:
    // the CTA-pair shrink / dH ([piece][CTA of the pair][256 columns][128 rows]) and dB / dA
    // (per cut item: [part][chunk][256 rows x 64 columns])
    P->off_partials = round_up(shadow, 1024);
    const size_t partials = std::max(static_cast<size_t>(P->win_units) * 2 * BM * 256 * 4,
                                     static_cast<size_t>(std::max(P->da_units, P->db_units)) * WG_UNIT * 4);
    P->off_himg = round_up(P->off_partials + partials, 1024);
    P->off_dhimg = P->off_himg + static_cast<size_t>(P->n_images) * IMG_BYTES;
    P->ws_bytes = P->off_dhimg + static_cast<size_t>(P->n_images) * IMG_BYTES;
    if (pr.dtype == MLORA_BF16_W4 && !P->w4_fused) {
      // the bf16 expansion of the 4-bit base, Wt [d_out, d_in]
      P->off_wexp = round_up(P->ws_bytes, 1024);
      P->ws_bytes = P->off_wexp + static_cast<size_t>(pr.d_out) * pr.d_in * 2;
    }
  } else {
    P->ws_bytes = 0;
  }
  // raster group for the base GEMMs: enough M tiles that one wave of CTAs shares W tiles
  P->group_m = 16;
}

template <typename T>
size_t table_bytes(const std::vector<T>& v) {
  return round_up(std::max<size_t>(1, v.size()) * sizeof(T), 256);
}

// Arrival counters of split items: 8 per split CTA-pair item (CTA of the pair x row quarter), then
// 8 per cut dA item and 8 per cut dB item (row quarter x 128-row half: one per epilogue warp).
size_t counter_ints(const mlora_plan_t* P) {
  return static_cast<size_t>(P->n_split) * 8 + static_cast<size_t>(P->da_sets) * 8 +
         static_cast<size_t>(P->db_sets) * 8;
}

mlora_status upload(mlora_plan_t* P) {
  cudaError_t e = cudaGetDevice(&P->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, P->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  const size_t b_segs = table_bytes(P->segs), b_mt = table_bytes(P->mtiles), b_it = table_bytes(P->img_tile),
               b_cs = table_bytes(P->col_sub), b_sc = table_bytes(P->col_scale), b_sub = table_bytes(P->subs),
               b_win = table_bytes(P->win), b_win2 = table_bytes(P->win2), b_da = table_bytes(P->da),
               b_db = table_bytes(P->db), b_daf = table_bytes(P->da_first), b_dbf = table_bytes(P->db_first),
               b_w2f = table_bytes(P->win2_first), b_w2d = table_bytes(P->win2d),
               b_w2df = table_bytes(P->win2d_first), b_adam = table_bytes(P->adam), b_err = 256,
               b_cnt = round_up(counter_ints(P) * sizeof(int), 256);
  const size_t total = b_segs + b_mt + b_it + b_cs + b_sc + b_sub + b_win + b_win2 + b_da + b_db + b_daf + b_dbf +
                       b_w2f + b_w2d + b_w2df + b_adam + b_err + b_cnt;
  e = cudaMalloc(&P->dev_block, total);
  if (e != cudaSuccess) {
    P->dev_block = nullptr;
    cudaGetLastError();
    return fail(MLORA_ERR_OOM, std::string("cudaMalloc of the plan tables failed: ") + cudaGetErrorString(e));
  }
  uint8_t* b = static_cast<uint8_t*>(P->dev_block);
  size_t o = 0;
  auto place = [&](auto*& dst, const auto& vec, size_t bytes) -> cudaError_t {
    using TT = std::remove_reference_t<decltype(*dst)>;
    dst = reinterpret_cast<TT*>(b + o);
    o += bytes;
    if (vec.empty()) return cudaSuccess;
    return cudaMemcpy(dst, vec.data(), vec.size() * sizeof(vec[0]), cudaMemcpyHostToDevice);
  };
  if ((e = place(P->d_segs, P->segs, b_segs)) != cudaSuccess ||
      (e = place(P->d_mtiles, P->mtiles, b_mt)) != cudaSuccess ||
      (e = place(P->d_img_tile, P->img_tile, b_it)) != cudaSuccess ||
      (e = place(P->d_col_sub, P->col_sub, b_cs)) != cudaSuccess ||
      (e = place(P->d_col_scale, P->col_scale, b_sc)) != cudaSuccess ||
      (e = place(P->d_subs, P->subs, b_sub)) != cudaSuccess ||
      (e = place(P->d_win, P->win, b_win)) != cudaSuccess || (e = place(P->d_win2, P->win2, b_win2)) != cudaSuccess ||
      (e = place(P->d_da, P->da, b_da)) != cudaSuccess || (e = place(P->d_db, P->db, b_db)) != cudaSuccess ||
      (e = place(P->d_da_first, P->da_first, b_daf)) != cudaSuccess ||
      (e = place(P->d_db_first, P->db_first, b_dbf)) != cudaSuccess ||
      (e = place(P->d_win2_first, P->win2_first, b_w2f)) != cudaSuccess ||
      (e = place(P->d_win2d, P->win2d, b_w2d)) != cudaSuccess ||
      (e = place(P->d_win2d_first, P->win2d_first, b_w2df)) != cudaSuccess ||
      (e = place(P->d_adam, P->adam, b_adam)) != cudaSuccess)
    return cuda_fail(e, "uploading the plan tables");
  P->d_err = reinterpret_cast<int*>(b + o);
  e = cudaMemset(P->d_err, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  o += b_err;
  if (counter_ints(P) > 0) {
    P->d_part_cnt = reinterpret_cast<int*>(b + o);
    e = cudaMemset(P->d_part_cnt, 0, counter_ints(P) * sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  }
  P->on_device = true;
  return MLORA_OK;
}

enum KernelId {
  K_PACK_FWD = 0, K_SHRINK, K_FWD_GEMM, K_PACK_BWD, K_H_IMAGES, K_DH, K_DB, K_BWD_GEMM, K_DA, K_ADAMW,
  K_F32_FWD, K_F32_BWD, K_W4_EXPAND, K_COUNT
};
const char* const kKernelNames[K_COUNT] = {
    "pack_fwd", "shrink", "fwd_gemm", "pack_bwd", "h_images", "dH", "dB", "bwd_gemm", "dA", "adamw",
    "f32_forward", "f32_backward", "w4_expand"};
// kernels launched by each id (a pack step is two kernels, the fp32 passes several)
const int kKernelLaunches[K_COUNT] = {2, 1, 1, 2, 1, 1, 1, 1, 1, 1, 2, 4, 1};   // pack steps are two kernels

std::atomic<long long> g_launches{0};

cudaEvent_t next_event(mlora_plan_t* P) {
  if (P->ev_next == P->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    P->ev_pool.push_back(e);
  }
  return P->ev_pool[P->ev_next++];
}

// Run one launch step; with profiling on, bracket it by events on the same stream.
template <typename F>
cudaError_t timed(const mlora_plan_t* Pc, int id, cudaStream_t s, F&& launch) {
  mlora_plan_t* P = const_cast<mlora_plan_t*>(Pc);
  cudaEvent_t a = nullptr, b = nullptr;
  if (P->profiling) {
    a = next_event(P);
    b = next_event(P);
    if (a && b) cudaEventRecord(a, s);
  }
  cudaError_t e = launch();
  if (e == cudaSuccess) g_launches += kKernelLaunches[id];
  if (a && b) {
    cudaEventRecord(b, s);
    P->ev_pending.push_back({id, {a, b}});
  }
  return e;
}

GemmArgs base_args(const mlora_plan_t* P) {
  GemmArgs g{};
  g.N = static_cast<int>(P->prob.n_tokens);
  g.d_in = P->prob.d_in;
  g.d_out = P->prob.d_out;
  g.n_mtiles = P->n_mtiles;
  g.group_m = P->group_m;
  g.mtiles = P->d_mtiles;
  g.win = P->d_win;
  g.segs = P->d_segs;
  if (P->grouped) {
    g.subs = P->d_subs;
    g.col_sub = P->d_col_sub;
    g.col_scale = P->d_col_scale;
    g.n_groups = P->n_groups;
  }
  g.err = P->d_err;
  g.timeout_ns = P->timeout_ns;
  g.pdl = P->pdl ? 1 : 0;
  return g;
}

int grid_of(const mlora_plan_t* P, int items) { return std::max(1, std::min(items, P->num_sms)); }

mlora_status check_exec(const mlora_plan_t* P) {
  if (!P) return fail(MLORA_ERR_INVALID, "null plan");
  if (!P->on_device) return fail(MLORA_ERR_INVALID, "plan was built with MLORA_PLAN_HOST_ONLY");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != P->device)
    return fail(MLORA_ERR_INVALID, "the current device is not the one the plan was built on");
  // Make the device's primary context current on this thread: a thread that has only selected
  // the device (an autograd worker, say) may not have it yet, and the tensor-map encoder needs it.
  cudaError_t e = cudaSetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  return MLORA_OK;
}

}  // namespace

extern "C" {

mlora_status mlora_plan_grouped(const mlora_problem* problem, const mlora_group* groups, int32_t n_groups,
                                const mlora_segment* segs, int32_t n_segs, size_t* workspace_bytes,
                                mlora_plan_t** out) {
  g_last_error.clear();
  if (!out || !workspace_bytes) return fail(MLORA_ERR_INVALID, "null output pointer");
  *out = nullptr;
  mlora_status st = validate(problem, groups, n_groups, segs, n_segs);
  if (st != MLORA_OK) return st;
  mlora_plan_t* P = new (std::nothrow) mlora_plan_s();
  if (!P) return fail(MLORA_ERR_OOM, "host allocation failed");
  P->prob = *problem;
  P->n_segs = n_segs;
  P->n_groups = n_groups;
  P->n_jobs = n_segs / n_groups;
  P->grouped = n_groups > 1;
  P->groups.assign(groups, groups + n_groups);
  P->user.assign(segs, segs + n_segs);
  if (problem->flags & MLORA_DEBUG_SHORT_TIMEOUT) P->timeout_ns = SHORT_TIMEOUT_NS;
  // Programmatic overlap of a kernel's prologue with its predecessor's tail saves a few microseconds
  // per launch, which only short kernels notice; with long ones it measured slower (one box,
  // alternating: the Llama-3-8B layer 83.5-83.9 against 82.1-82.7 ms per step, the many-small-jobs
  // pack 12.66-12.77 against 12.51-12.54 ms, mlp_up 0.6 % and the shared q/k/v pack even; q_proj,
  // 2.7e11 multiply-adds per base product, 0.738-0.740 against 0.751-0.755 ms).  It is kept for
  // plans whose base product N d_in d_out is at most 4e11.
  if (static_cast<double>(problem->n_tokens) * problem->d_in * problem->d_out > 4e11) P->pdl = false;
  if (problem->flags & MLORA_OVERLAP) P->pdl = true;
  if (problem->flags & MLORA_NO_OVERLAP) P->pdl = false;
  if (problem->flags & MLORA_REUSE_STAGING) P->reuse_staging = true;
  if (problem->flags & MLORA_W4_FUSED) P->w4_fused = true;
  // the copy-withholding test hook is honoured only with the 1 ms wait limit
  if ((problem->flags & MLORA_DEBUG_DROP_COPY) && (problem->flags & MLORA_DEBUG_SHORT_TIMEOUT)) P->debug_drop = true;
  if ((problem->flags & MLORA_DEBUG_DROP_COPY_PAIRS) && (problem->flags & MLORA_DEBUG_SHORT_TIMEOUT))
    P->debug_drop_pairs = true;
  if (!(problem->flags & MLORA_PLAN_HOST_ONLY)) {
    // the planner sizes the last wave of the CTA-pair work lists for this device's SM count
    cudaError_t e = cudaGetDevice(&P->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, P->device);
    if (e != cudaSuccess) {
      mlora_plan_destroy(P);
      return cuda_fail(e, "querying the device");
    }
  }
  build_tables(P);
  if (problem->mem_budget_bytes > 0) {
    mlora_memory m{};
    mlora_memory_estimate(P, &m);
    if (m.total > problem->mem_budget_bytes) {
      char buf[200];
      snprintf(buf, sizeof buf, "the pack needs %lld bytes of device memory, more than the budget of %lld",
               static_cast<long long>(m.total), static_cast<long long>(problem->mem_budget_bytes));
      mlora_plan_destroy(P);
      return fail(MLORA_ERR_OOM, buf);
    }
  }
  if (!(problem->flags & MLORA_PLAN_HOST_ONLY)) {
    st = upload(P);
    if (st != MLORA_OK) {
      mlora_plan_destroy(P);
      return st;
    }
  }
  *workspace_bytes = P->ws_bytes;
  *out = P;
  return MLORA_OK;
}

mlora_status mlora_plan(const mlora_problem* problem, const mlora_segment* segs, int32_t n_segs,
                        size_t* workspace_bytes, mlora_plan_t** out) {
  if (!problem) return fail(MLORA_ERR_INVALID, "null problem, group or segment table");
  const mlora_group all{0, problem->d_out};
  return mlora_plan_grouped(problem, &all, 1, segs, n_segs, workspace_bytes, out);
  return MLORA_OK;
}

void mlora_plan_destroy(mlora_plan_t* plan) {
  if (!plan) return;
  for (cudaEvent_t e : plan->ev_pool) cudaEventDestroy(e);
  if (plan->dev_block) cudaFree(plan->dev_block);
  delete plan;
}

int64_t mlora_h_elems(const mlora_plan_t* plan) { return plan ? plan->h_elems : -1; }

}  // extern "C"

namespace {

// Forward of any dtype: Wt for bf16 / fp32 plans, (Wq, Ws) for 4-bit-base plans.
mlora_status forward_impl(const mlora_plan_t* P, const void* X, const void* Wt, const void* Wq, const float* Ws, void* Y,
                          float* H, void* workspace, void* stream) {
  g_last_error.clear();
  mlora_status st = check_exec(P);
  if (st != MLORA_OK) return st;
  const bool w4 = P->prob.dtype == MLORA_BF16_W4;
  if (w4 != (Wt == nullptr))
    return fail(MLORA_ERR_INVALID, w4 ? "this plan has a 4-bit base: use mlora_forward_w4"
                                      : "this plan has a bf16/fp32 base: use mlora_forward");
  const void* Wany = w4 ? Wq : Wt;
  if (!X || !Wany || !Y || (w4 && !Ws) || (!H && P->h_elems > 0)) return fail(MLORA_ERR_INVALID, "null tensor argument");
  if (!aligned16(X) || !aligned16(Wany) || !aligned16(Y) || !aligned16(H) || !aligned16(Ws))
    return fail(MLORA_ERR_INVALID, "X, the base weight, Y and H must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const mlora_problem& pr = P->prob;
  cudaError_t e;
  if (pr.dtype == MLORA_F32) {
    e = timed(P, K_F32_FWD, s, [&] { return launch_f32_forward(P->d_segs, P->n_jobs, pr.n_tokens, pr.d_in, pr.d_out, P->h_elems,
                           P->max_rank, P->max_tokens, P->num_sms, static_cast<const float*>(X), static_cast<const float*>(Wt), static_cast<float*>(Y), H, s); });
    return e == cudaSuccess ? MLORA_OK : cuda_fail(e, "fp32 forward launch");
  }
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(MLORA_ERR_INVALID, "workspace must be a 256-byte aligned device buffer");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* at_all = reinterpret_cast<__nv_bfloat16*>(ws + P->off_shadow);
  __nv_bfloat16* bt_all =
      reinterpret_cast<__nv_bfloat16*>(ws + P->off_shadow + round_up(static_cast<size_t>(P->C_total) * pr.d_in * 2, 1024));
  uint8_t* himg = ws + P->off_himg;

  // A 4-bit base is expanded once into the workspace (then everything below is the bf16 path),
  // unless the plan asked for the GEMMs that expand it in shared memory.
  const bool fused4 = w4 && P->w4_fused;
  if (w4 && !fused4) {
    __nv_bfloat16* wexp = reinterpret_cast<__nv_bfloat16*>(ws + P->off_wexp);
    e = timed(P, K_W4_EXPAND, s, [&] { return launch_w4_expand(Wq, Ws, wexp, pr.d_in, pr.d_out, P->num_sms, s, P->pdl); });
    if (e != cudaSuccess) return cuda_fail(e, "4-bit expansion launch");
    Wt = wexp;
  }
  // With MLORA_REUSE_STAGING the shadows are not rebuilt when this workspace already holds them
  // for the current masters (written by the last forward, or refreshed by mlora_adamw_ws).
  if (!(P->reuse_staging && P->shadows_valid && P->shadows_ws == workspace)) {
    e = timed(P, K_PACK_FWD, s, [&] { return launch_pack_fwd(P->d_subs, P->d_col_sub, P->C_total, pr.d_in, pr.d_out, at_all, bt_all, P->num_sms, s, P->pdl); });
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
  }

  const bool pairs = !(pr.flags & MLORA_GEMM_SINGLE_CTA);
  CUtensorMap mX, mAt, mW, mBt, mI, mQ, mS, mW64, mBt64;
  if ((st = make_map(&mX, X, pr.d_in, pr.n_tokens, pr.d_in, 64, 128)) != MLORA_OK) return st;
  if ((st = make_map(&mAt, at_all, pr.d_in, P->C_total, pr.d_in, 64, 64)) != MLORA_OK) return st;
  if (fused4) {
    // codes [d_out, d_in/2] bytes, box 32 bytes x 128 rows; scales [d_in/64, d_out], box 128 x 1
    if ((st = make_map_plain(&mQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, pr.d_in / 2, pr.d_out, pr.d_in / 2, 32, 128)) !=
        MLORA_OK)
      return st;
    if ((st = make_map_plain(&mS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Ws, pr.d_out, pr.d_in / 64, pr.d_out, 128, 1)) !=
        MLORA_OK)
      return st;
  } else if ((st = make_map(&mW, Wt, pr.d_in, pr.d_out, pr.d_in, 64, pairs ? 128 : 256)) != MLORA_OK) {
    return st;
  }
  if ((st = make_map(&mBt, bt_all, P->C_total, pr.d_out, P->C_total, 64, pairs ? 128 : 256)) != MLORA_OK) return st;
  if (pairs && !fused4) {   // 64-row boxes of the same tensors for half-width tail tiles
    if ((st = make_map(&mW64, Wt, pr.d_in, pr.d_out, pr.d_in, 64, 64)) != MLORA_OK) return st;
    if ((st = make_map(&mBt64, bt_all, P->C_total, pr.d_out, P->C_total, 64, 64)) != MLORA_OK) return st;
  }
  if ((st = make_map(&mI, himg, CHUNK_COLS, P->n_images * BM, CHUNK_COLS, 64, 128)) != MLORA_OK) return st;

  GemmArgs g = base_args(P);
  g.kmain = (pr.d_in + BK - 1) / BK;
  g.img_out = himg;
  g.hout = H;
  if (P->win_pairs) {
    g.win = P->d_win2;
    g.n_items = static_cast<int>(P->win2.size());
    g.debug_drop = P->debug_drop_pairs ? 1 : 0;
    g.cta_first = P->d_win2_first;
    g.partials = P->n_split ? reinterpret_cast<float*>(ws + P->off_partials) : nullptr;
    g.part_cnt = P->d_part_cnt;
    const int n_pairs = static_cast<int>(P->win2_first.size()) - 1;
    e = timed(P, K_SHRINK, s, [&] { return launch_win_2sm<MODE_SHRINK>(mX, mAt, g, n_pairs, s); });
  } else {
    g.n_items = static_cast<int>(P->win.size());
    g.debug_drop = P->debug_drop ? 1 : 0;
    e = timed(P, K_SHRINK, s, [&] { return launch_seg_gemm<MODE_SHRINK>(mX, mAt, mAt, mX, g, grid_of(P, g.n_items), s); });
  }
  if (e != cudaSuccess) return cuda_fail(e, "shrink launch");

  g = base_args(P);
  g.kmain = (pr.d_in + BK - 1) / BK;
  g.n_tiles_n = (pr.d_out + BN - 1) / BN;
  g.out = Y;
  g.ld_out = pr.d_out;
  if (pairs || fused4) set_raster(g, pr.d_in);   // the single-CTA engine keeps its M-tile groups
  if (fused4) {
    g.n_items = ((P->n_mtiles + 1) / 2) * g.n_tiles_n;
    e = timed(P, K_FWD_GEMM, s, [&] {
      return launch_gemm_2sm_w4<MODE_FWD>(mX, mQ, mS, mBt, mI, g, std::max(1, std::min(g.n_items, P->num_sms / 2)), s);
    });
  } else if (pairs) {
    const int n_pairs = pair_gemm_items(P->n_mtiles, P->num_sms, g);
    g.debug_drop = P->debug_drop_pairs ? 1 : 0;
    CUtensorMap mY;
    if ((st = make_map(&mY, Y, pr.d_out, pr.n_tokens, pr.d_out, 64, 128)) != MLORA_OK) return st;
    e = timed(P, K_FWD_GEMM, s, [&] { return launch_gemm_2sm<MODE_FWD>(mX, mW, mBt, mI, mW64, mBt64, mY, g, n_pairs, s); });
  } else {
    g.n_items = P->n_mtiles * g.n_tiles_n;
    e = timed(P, K_FWD_GEMM, s, [&] { return launch_seg_gemm<MODE_FWD>(mX, mW, mBt, mI, g, grid_of(P, g.n_items), s); });
  }
  if (e != cudaSuccess) return cuda_fail(e, "forward GEMM launch");
  {
    mlora_plan_t* Pm = const_cast<mlora_plan_t*>(P);
    Pm->staged_valid = true;
    Pm->staged_ws = workspace;
    Pm->staged_H = H;
    Pm->shadows_valid = true;
    Pm->shadows_ws = workspace;
    Pm->staged_wq = w4 && !fused4 ? Wq : nullptr;
    Pm->staged_wscale = w4 && !fused4 ? Ws : nullptr;
  }
  return MLORA_OK;
}

// Backward of any dtype (see forward_impl).
mlora_status backward_impl(const mlora_plan_t* P, const void* X, const void* Wt, const void* Wq, const float* Ws,
                           const void* dY, const float* H, void* dX, float* dH, void* workspace, void* stream) {
  g_last_error.clear();
  mlora_status st = check_exec(P);
  if (st != MLORA_OK) return st;
  if (!P->can_backward) return fail(MLORA_ERR_INVALID, "the plan's segments have no dAt/dBt buffers");
  const bool w4 = P->prob.dtype == MLORA_BF16_W4;
  if (w4 != (Wt == nullptr))
    return fail(MLORA_ERR_INVALID, w4 ? "this plan has a 4-bit base: use mlora_backward_w4"
                                      : "this plan has a bf16/fp32 base: use mlora_backward");
  const void* Wany = w4 ? Wq : Wt;
  if (!X || !Wany || !dY || !dX || (w4 && !Ws) || ((!H || !dH) && P->h_elems > 0))
    return fail(MLORA_ERR_INVALID, "null tensor argument");
  if (!aligned16(X) || !aligned16(Wany) || !aligned16(dY) || !aligned16(dX) || !aligned16(H) || !aligned16(dH) ||
      !aligned16(Ws))
    return fail(MLORA_ERR_INVALID, "X, the base weight, dY, dX, H and dH must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const mlora_problem& pr = P->prob;
  cudaError_t e;
  if (pr.dtype == MLORA_F32) {
    e = timed(P, K_F32_BWD, s, [&] { return launch_f32_backward(P->d_segs, P->n_jobs, pr.n_tokens, pr.d_in, pr.d_out, P->h_elems, P->max_rank, P->max_tokens, P->num_sms,
                            static_cast<const float*>(X), static_cast<const float*>(Wt), static_cast<const float*>(dY),
                            H, static_cast<float*>(dX), dH, s); });
    return e == cudaSuccess ? MLORA_OK : cuda_fail(e, "fp32 backward launch");
  }
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(MLORA_ERR_INVALID, "workspace must be a 256-byte aligned device buffer");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* at_all = reinterpret_cast<__nv_bfloat16*>(ws + P->off_shadow);
  __nv_bfloat16* bt_all =
      reinterpret_cast<__nv_bfloat16*>(ws + P->off_shadow + round_up(static_cast<size_t>(P->C_total) * pr.d_in * 2, 1024));
  uint8_t* himg = ws + P->off_himg;
  uint8_t* dhimg = ws + P->off_dhimg;

  // The backward reads the same two bf16 shadows as the forward, At_all [C, d_in] and
  // Bt_all [d_out, C], as MN-major operands, and the staged s*H images.  With
  // MLORA_REUSE_STAGING, when this workspace and H are the ones the last forward used (and no
  // AdamW step ran since), they are still in place and are not rebuilt.
  const bool reuse = P->reuse_staging && P->staged_valid && P->staged_ws == workspace && P->staged_H == H;
  const bool fused4 = w4 && P->w4_fused;
  if (w4 && !fused4) {
    // the bf16 expansion of the 4-bit base; with reuse, the forward's is still in place when it
    // expanded the same codes and scales
    __nv_bfloat16* wexp = reinterpret_cast<__nv_bfloat16*>(ws + P->off_wexp);
    if (!(reuse && P->staged_wq == Wq && P->staged_wscale == Ws)) {
      e = timed(P, K_W4_EXPAND, s, [&] { return launch_w4_expand(Wq, Ws, wexp, pr.d_in, pr.d_out, P->num_sms, s, P->pdl); });
      if (e != cudaSuccess) return cuda_fail(e, "4-bit expansion launch");
    }
    Wt = wexp;
  }
  if (!reuse) {
    e = timed(P, K_PACK_BWD, s, [&] { return launch_pack_fwd(P->d_subs, P->d_col_sub, P->C_total, pr.d_in, pr.d_out, at_all, bt_all, P->num_sms, s, P->pdl); });
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    mlora_plan_t* Pm = const_cast<mlora_plan_t*>(P);
    Pm->shadows_valid = true;
    Pm->shadows_ws = workspace;
    e = timed(P, K_H_IMAGES, s, [&] { return launch_h_images(P->d_segs, P->d_col_scale, P->d_mtiles, P->d_img_tile, static_cast<int>(P->n_images), pr.n_tokens, H, himg, s, P->pdl); });
    if (e != cudaSuccess) return cuda_fail(e, "image launch");
  }

  const bool pairs = !(pr.flags & MLORA_GEMM_SINGLE_CTA);
  CUtensorMap mdY, mdYt, mBt64, mWmn, mAt64, mXt, mHi, mdHi, mdHi64, mQ, mS;
  if ((st = make_map(&mdY, dY, pr.d_out, pr.n_tokens, pr.d_out, 64, 128)) != MLORA_OK) return st;
  if ((st = make_map(&mdYt, dY, pr.d_out, pr.n_tokens, pr.d_out, 64, 64)) != MLORA_OK) return st;
  if ((st = make_map(&mBt64, bt_all, P->C_total, pr.d_out, P->C_total, 64, 64)) != MLORA_OK) return st;
  if (fused4) {
    // codes: 64 rows (d_out) x 64 bytes (128 d_in); scales: 64 (d_out) x 2 groups (d_in)
    if ((st = make_map_plain(&mQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Wq, pr.d_in / 2, pr.d_out, pr.d_in / 2, 64, 64)) !=
        MLORA_OK)
      return st;
    if ((st = make_map_plain(&mS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Ws, pr.d_out, pr.d_in / 64, pr.d_out, 64, 2)) !=
        MLORA_OK)
      return st;
  } else if ((st = make_map(&mWmn, Wt, pr.d_in, pr.d_out, pr.d_in, 64, 64)) != MLORA_OK) {
    return st;
  }
  if ((st = make_map(&mAt64, at_all, pr.d_in, P->C_total, pr.d_in, 64, 64)) != MLORA_OK) return st;
  if ((st = make_map(&mXt, X, pr.d_in, pr.n_tokens, pr.d_in, 64, 64)) != MLORA_OK) return st;
  if ((st = make_map(&mHi, himg, CHUNK_COLS, P->n_images * BM, CHUNK_COLS, 64, 64)) != MLORA_OK) return st;
  if ((st = make_map(&mdHi, dhimg, CHUNK_COLS, P->n_images * BM, CHUNK_COLS, 64, 128)) != MLORA_OK) return st;
  if ((st = make_map(&mdHi64, dhimg, CHUNK_COLS, P->n_images * BM, CHUNK_COLS, 64, 64)) != MLORA_OK) return st;

  // dH = s dY B^T  (+ staged dHtilde images)
  GemmArgs g = base_args(P);
  g.kmain = (pr.d_out + BK - 1) / BK;
  g.img_out = dhimg;
  g.hout = dH;
  if (P->win_pairs) {
    g.win = P->d_win2d;
    g.n_items = static_cast<int>(P->win2d.size());
    g.cta_first = P->d_win2d_first;
    g.partials = P->n_split ? reinterpret_cast<float*>(ws + P->off_partials) : nullptr;
    g.part_cnt = P->d_part_cnt;
    const int n_pairs = static_cast<int>(P->win2d_first.size()) - 1;
    e = timed(P, K_DH, s, [&] { return launch_win_2sm<MODE_DH>(mdY, mBt64, g, n_pairs, s); });
  } else {
    g.n_items = static_cast<int>(P->win.size());
    e = timed(P, K_DH, s, [&] { return launch_seg_gemm<MODE_DH>(mdY, mBt64, mBt64, mdY, g, grid_of(P, g.n_items), s); });
  }
  if (e != cudaSuccess) return cuda_fail(e, "dH launch");

  // dB = Htilde^T dY
  g = base_args(P);
  g.witems = P->d_db;
  g.n_items = static_cast<int>(P->db.size());
  g.cta_first = P->d_db_first;
  g.partials = reinterpret_cast<float*>(ws + P->off_partials);
  g.part_cnt = P->d_part_cnt ? P->d_part_cnt + static_cast<size_t>(P->n_split) * 8 + static_cast<size_t>(P->da_sets) * 8
                             : nullptr;
  const int db_ctas = static_cast<int>(P->db_first.size()) - 1;
  e = timed(P, K_DB, s, [&] { return launch_seg_gemm<MODE_DB>(mdYt, mdYt, mdYt, mHi, g, db_ctas, s); });
  if (e != cudaSuccess) return cuda_fail(e, "dB launch");

  // dX = dY W^T + dHtilde A^T
  g = base_args(P);
  g.kmain = (pr.d_out + BK - 1) / BK;
  g.n_tiles_n = (pr.d_in + BN - 1) / BN;
  g.out = dX;
  g.ld_out = pr.d_in;
  if (pairs || fused4) set_raster(g, pr.d_out);   // the single-CTA engine keeps its M-tile groups
  if (fused4) {
    g.n_items = ((P->n_mtiles + 1) / 2) * g.n_tiles_n;
    e = timed(P, K_BWD_GEMM, s, [&] {
      return launch_gemm_2sm_w4<MODE_BWD>(mdY, mQ, mS, mAt64, mdHi, g, std::max(1, std::min(g.n_items, P->num_sms / 2)), s);
    });
  } else if (pairs) {
    const int n_pairs = pair_gemm_items(P->n_mtiles, P->num_sms, g);
    CUtensorMap mdX;
    if ((st = make_map(&mdX, dX, pr.d_in, pr.n_tokens, pr.d_in, 64, 128)) != MLORA_OK) return st;
    e = timed(P, K_BWD_GEMM, s, [&] {
      return launch_gemm_2sm<MODE_BWD>(mdY, mWmn, mAt64, mdHi, mWmn, mAt64, mdX, g, n_pairs, s);
    });
  } else {
    g.n_items = P->n_mtiles * g.n_tiles_n;
    e = timed(P, K_BWD_GEMM, s, [&] { return launch_seg_gemm<MODE_BWD>(mdY, mWmn, mAt64, mdHi, g, grid_of(P, g.n_items), s); });
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward GEMM launch");

  // dA = X^T dHtilde
  g = base_args(P);
  g.witems = P->d_da;
  g.n_items = static_cast<int>(P->da.size());
  g.cta_first = P->d_da_first;
  g.partials = reinterpret_cast<float*>(ws + P->off_partials);
  g.part_cnt = P->d_part_cnt ? P->d_part_cnt + static_cast<size_t>(P->n_split) * 8 : nullptr;
  const int da_ctas = static_cast<int>(P->da_first.size()) - 1;
  e = timed(P, K_DA, s, [&] { return launch_seg_gemm<MODE_DA>(mXt, mXt, mXt, mdHi64, g, da_ctas, s); });
  if (e != cudaSuccess) return cuda_fail(e, "dA launch");
  return MLORA_OK;
}

}  // namespace

extern "C" {

mlora_status mlora_forward(const mlora_plan_t* P, const void* X, const void* Wt, void* Y, float* H, void* workspace,
                           void* stream) {
  if (!Wt) return fail(MLORA_ERR_INVALID, "null tensor argument");
  return forward_impl(P, X, Wt, nullptr, nullptr, Y, H, workspace, stream);
}

mlora_status mlora_forward_w4(const mlora_plan_t* P, const void* X, const void* Wq, const float* Wscale, void* Y,
                              float* H, void* workspace, void* stream) {
  if (!Wq || !Wscale) return fail(MLORA_ERR_INVALID, "null tensor argument");
  return forward_impl(P, X, nullptr, Wq, Wscale, Y, H, workspace, stream);
}

mlora_status mlora_backward(const mlora_plan_t* P, const void* X, const void* Wt, const void* dY, const float* H,
                            void* dX, float* dH, void* workspace, void* stream) {
  if (!Wt) return fail(MLORA_ERR_INVALID, "null tensor argument");
  return backward_impl(P, X, Wt, nullptr, nullptr, dY, H, dX, dH, workspace, stream);
}

mlora_status mlora_backward_w4(const mlora_plan_t* P, const void* X, const void* Wq, const float* Wscale,
                               const void* dY, const float* H, void* dX, float* dH, void* workspace, void* stream) {
  if (!Wq || !Wscale) return fail(MLORA_ERR_INVALID, "null tensor argument");
  return backward_impl(P, X, nullptr, Wq, Wscale, dY, H, dX, dH, workspace, stream);
}

}  // extern "C"

namespace {

mlora_status adamw_impl(const mlora_plan_t* P, float lr, float beta1, float beta2, float eps, float weight_decay,
                        int32_t step, void* workspace, void* stream) {
  g_last_error.clear();
  mlora_status st = check_exec(P);
  if (st != MLORA_OK) return st;
  if (!P->can_adamw) return fail(MLORA_ERR_INVALID, "the plan's segments lack gradient or moment buffers");
  if (step < 1) return fail(MLORA_ERR_INVALID, "step must be >= 1");
  if (!(beta1 >= 0.f && beta1 < 1.f && beta2 >= 0.f && beta2 < 1.f) || !std::isfinite(lr) || !std::isfinite(eps) ||
      !std::isfinite(weight_decay))
    return fail(MLORA_ERR_INVALID, "bad AdamW hyper-parameters");
  const bool refresh = workspace != nullptr && P->prob.dtype != MLORA_F32;
  if (refresh && (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(MLORA_ERR_INVALID, "workspace must be a 256-byte aligned device buffer");
  mlora_plan_t* Pm = const_cast<mlora_plan_t*>(P);
  Pm->staged_valid = false;   // the masters change: the backward's staging is stale
  Pm->shadows_valid = false;
  __nv_bfloat16* at_all = nullptr;
  __nv_bfloat16* bt_all = nullptr;
  if (refresh) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    at_all = reinterpret_cast<__nv_bfloat16*>(ws + P->off_shadow);
    bt_all = reinterpret_cast<__nv_bfloat16*>(
        ws + P->off_shadow + round_up(static_cast<size_t>(P->C_total) * P->prob.d_in * 2, 1024));
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed(P, K_ADAMW, s, [&] {
    return launch_adamw(P->d_adam, static_cast<int>(P->adam.size()), lr, beta1, beta2, eps, weight_decay, step,
                        P->num_sms, s, P->pdl, at_all, bt_all, P->C_total);
  });
  if (e != cudaSuccess) return cuda_fail(e, "AdamW launch");
  if (refresh) {
    // Only the adapters' columns were written: the padding of the packed space must already be
    // zero, which holds when a forward or backward packed this workspace before.
    Pm->shadows_valid = P->shadows_ws == workspace;
  }
  return MLORA_OK;
}

}  // namespace

extern "C" {

mlora_status mlora_adamw(const mlora_plan_t* P, float lr, float beta1, float beta2, float eps, float weight_decay,
                         int32_t step, void* stream) {
  return adamw_impl(P, lr, beta1, beta2, eps, weight_decay, step, nullptr, stream);
}

mlora_status mlora_adamw_ws(const mlora_plan_t* P, float lr, float beta1, float beta2, float eps,
                            float weight_decay, int32_t step, void* workspace, void* stream) {
  if (!workspace) return fail(MLORA_ERR_INVALID, "null workspace");
  return adamw_impl(P, lr, beta1, beta2, eps, weight_decay, step, workspace, stream);
}

mlora_status mlora_sync_status(const mlora_plan_t* P, void* stream) {
  g_last_error.clear();
  mlora_status st = check_exec(P);
  if (st != MLORA_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, P->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (v != 0) {
    e = cudaMemset(P->d_err, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    // a launch that gave up may have left split items' arrival counts behind
    if (P->d_part_cnt) {
      e = cudaMemset(P->d_part_cnt, 0, counter_ints(P) * sizeof(int));
      if (e != cudaSuccess) return cuda_fail(e, "clearing the split items' counters");
    }
    char buf[96];
    snprintf(buf, sizeof buf, "a device-side wait gave up (code 0x%x)", v);
    return fail(MLORA_ERR_TIMEOUT, buf);
  }
  return MLORA_OK;
}

mlora_status mlora_plan_describe(const mlora_plan_t* P, int32_t what, int64_t* out, int64_t cap, int64_t* count) {
  if (!P || !count) return fail(MLORA_ERR_INVALID, "null plan or count");
  std::vector<int64_t> v;
  switch (what) {
    case MLORA_Q_SUMMARY:
      v = {P->prob.n_tokens, P->prob.d_in, P->prob.d_out, P->n_segs, P->n_mtiles, P->C_total, P->n_chunks,
           P->n_images, static_cast<int64_t>(P->win.size()), static_cast<int64_t>(P->da.size()),
           static_cast<int64_t>(P->db.size()), static_cast<int64_t>(P->ws_bytes)};
      break;
    case MLORA_Q_MTILES:
      for (const MTile& m : P->mtiles) v.insert(v.end(), {m.seg_first, m.seg_last, m.q_lo, m.nch, m.img_off});
      break;
    case MLORA_Q_COLUMNS:
      for (const DevSeg& d : P->segs) v.insert(v.end(), {d.c, d.rp});
      break;
    case MLORA_Q_WGRAD_A:
    case MLORA_Q_WGRAD_B: {
      const bool a = what == MLORA_Q_WGRAD_A;
      const std::vector<WItem>& it = a ? P->da : P->db;
      const std::vector<int>& first = a ? P->da_first : P->db_first;
      for (size_t c = 0; c + 1 < first.size(); ++c)
        for (int k = first[c]; k < first[c + 1]; ++k) {
          const WItem& w = it[k];
          v.insert(v.end(), {w.row0, w.seg, w.ga, w.gb, w.q0, w.nq, w.part, w.nparts, static_cast<int64_t>(c)});
        }
      break;
    }
    case MLORA_Q_WINDOW:
      for (const WinItem& w : P->win) v.insert(v.end(), {w.tile, w.q0, w.nq, w.dh_kb0, w.dh_nkb});
      break;
    case MLORA_Q_WINDOW_PAIRS: {
      v.push_back(P->win_pairs ? 1 : 0);
      const int kin = (P->prob.d_in + BK - 1) / BK;
      for (int prod = 0; prod < 2; ++prod) {
        const std::vector<WinItem>& it = prod ? P->win2d : P->win2;
        const std::vector<int>& first = prod ? P->win2d_first : P->win2_first;
        for (size_t p = 0; p + 1 < first.size(); ++p)
          for (int k = first[p]; k < first[p + 1]; ++k) {
            const WinItem& w = it[k];
            int k0, nk;
            win_krange(w, prod == 1, kin, k0, nk);
            v.insert(v.end(), {prod, static_cast<int64_t>(p), w.tile, w.q0, w.nq, k0, nk, w.part, w.nparts});
          }
      }
      break;
    }
    case MLORA_Q_ADAPTERS:
      for (const DevSub& sb : P->subs) v.insert(v.end(), {sb.job, sb.c0, sb.r, sb.o_lo, sb.o_hi});
      break;
    case MLORA_Q_GEMM_FWD:
    case MLORA_Q_GEMM_BWD: {
      // the CTA-pair base GEMM's work list exactly as the kernels decode it
      const bool fwd = what == MLORA_Q_GEMM_FWD;
      GemmArgs g = base_args(P);
      g.n_tiles_n = ((fwd ? P->prob.d_out : P->prob.d_in) + BN - 1) / BN;
      set_raster(g, fwd ? P->prob.d_in : P->prob.d_out);
      const int n_pairs = pair_gemm_items(P->n_mtiles, P->num_sms, g);
      v = {g.raster_n, g.group_m, g.n_items, g.n_full_items, n_pairs};
      for (int it = 0; it < g.n_items; ++it) {
        int mp, col0, width;
        pair::decode_item(g, it, mp, col0, width);
        v.insert(v.end(), {mp, col0, width});
      }
      break;
    }
    default:
      return fail(MLORA_ERR_INVALID, "unknown table");
  }
  *count = static_cast<int64_t>(v.size());
  if (out) std::copy(v.begin(), v.begin() + std::min<int64_t>(cap, *count), out);
  return MLORA_OK;
}

mlora_status mlora_profile_enable(mlora_plan_t* P, int32_t enable) {
  if (!P) return fail(MLORA_ERR_INVALID, "null plan");
  P->profiling = enable != 0;
  return MLORA_OK;
}

mlora_status mlora_profile_read(mlora_plan_t* P, double* ms, int64_t* launches, int32_t cap, int32_t* n_kernels) {
  if (!P || !n_kernels) return fail(MLORA_ERR_INVALID, "null plan or count");
  *n_kernels = K_COUNT;
  std::vector<double> acc(K_COUNT, 0.0);
  std::vector<int64_t> cnt(K_COUNT, 0);
  for (auto& pe : P->ev_pending) {
    cudaError_t e = cudaEventSynchronize(pe.second.second);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float t = 0.f;
    e = cudaEventElapsedTime(&t, pe.second.first, pe.second.second);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    acc[pe.first] += t;
    cnt[pe.first] += 1;
  }
  P->ev_pending.clear();
  P->ev_next = 0;
  for (int i = 0; i < K_COUNT && i < cap; ++i) {
    if (ms) ms[i] = acc[i];
    if (launches) launches[i] = cnt[i];
  }
  return MLORA_OK;
}

const char* mlora_kernel_name(int32_t id) { return (id >= 0 && id < K_COUNT) ? kKernelNames[id] : ""; }

int64_t mlora_launch_count(void) { return g_launches; }

mlora_status mlora_memory_estimate(const mlora_plan_t* P, mlora_memory* out) {
  if (!P || !out) return fail(MLORA_ERR_INVALID, "null plan or output");
  const mlora_problem& pr = P->prob;
  const int64_t e = pr.dtype == MLORA_F32 ? 4 : 2;
  int64_t params = 0;
  for (const DevSub& sb : P->subs) params += static_cast<int64_t>(sb.r) * (pr.d_in + (sb.o_hi - sb.o_lo));
  mlora_memory m{};
  m.base_weight = pr.dtype == MLORA_BF16_W4
                      ? static_cast<int64_t>(pr.d_in) * pr.d_out / 2 + static_cast<int64_t>(pr.d_in / 64) * pr.d_out * 4
                      : static_cast<int64_t>(pr.d_in) * pr.d_out * e;
  m.activations = 2 * pr.n_tokens * (static_cast<int64_t>(pr.d_in) + pr.d_out) * e;
  m.lora_params = params * 4;
  m.lora_grad_state = 3 * m.lora_params;
  m.lora_act = 2 * P->h_elems * 4;
  m.workspace = static_cast<int64_t>(P->ws_bytes);
  m.plan_tables = static_cast<int64_t>(table_bytes(P->segs) + table_bytes(P->mtiles) + table_bytes(P->img_tile) +
                                       table_bytes(P->col_sub) + table_bytes(P->col_scale) +
                                       table_bytes(P->subs) + table_bytes(P->win) + table_bytes(P->win2) +
                                       table_bytes(P->da) + table_bytes(P->db) + table_bytes(P->da_first) +
                                       table_bytes(P->db_first) + table_bytes(P->win2_first) +
                                       table_bytes(P->win2d) + table_bytes(P->win2d_first) +
                                       table_bytes(P->adam) + 256 +
                                       round_up(counter_ints(P) * sizeof(int), 256));
  m.total = m.base_weight + m.activations + m.lora_params + m.lora_grad_state + m.lora_act + m.workspace +
            m.plan_tables;
  *out = m;
  return MLORA_OK;
}

mlora_status mlora_cost_estimate(const mlora_plan_t* P, const mlora_cost_point* table, int32_t n_points,
                                 double* step_ms, int32_t* basis) {
  if (!P || !table || !step_ms || n_points < 1) return fail(MLORA_ERR_INVALID, "null plan, table or output");
  if (P->prob.dtype == MLORA_F32) return fail(MLORA_ERR_UNSUPPORTED, "the cost table covers bf16 packs");
  for (int i = 0; i < n_points; ++i)
    if (!(table[i].step_ms > 0.0) || table[i].n_tokens < 1 || table[i].d_in < 1 || table[i].d_out < 1)
      return fail(MLORA_ERR_INVALID, "cost table point with a non-positive size or time");
  auto work = [](double n, double din, double dout, double lora) { return 4.0 * n * din * dout + 6.0 * lora; };
  double lora = 0.0;
  for (const DevSub& sb : P->subs)
    lora += static_cast<double>(P->segs[sb.job].n) * sb.r * (P->prob.d_in + (sb.o_hi - sb.o_lo));
  const double F = work(static_cast<double>(P->prob.n_tokens), P->prob.d_in, P->prob.d_out, lora);
  // the points of this shape, by work
  std::vector<std::pair<double, double>> pts;   // (F, ms)
  for (int i = 0; i < n_points; ++i)
    if (table[i].d_in == P->prob.d_in && table[i].d_out == P->prob.d_out)
      pts.push_back({work(static_cast<double>(table[i].n_tokens), table[i].d_in, table[i].d_out, table[i].lora_work),
                     table[i].step_ms});
  std::sort(pts.begin(), pts.end());
  int b = 0;
  double t;
  if (pts.empty()) {
    // another shape's rate: the point whose work is nearest in ratio
    double best = 0.0, rate = 0.0;
    for (int i = 0; i < n_points; ++i) {
      const double f = work(static_cast<double>(table[i].n_tokens), table[i].d_in, table[i].d_out, table[i].lora_work);
      const double d = std::fabs(std::log(f / F));
      if (i == 0 || d < best) {
        best = d;
        rate = f / table[i].step_ms;
      }
    }
    t = F / rate;
    b = 2;
  } else if (F <= pts.front().first) {
    t = F / (pts.front().first / pts.front().second);
    b = F == pts.front().first ? 0 : 1;
  } else if (F >= pts.back().first) {
    t = F / (pts.back().first / pts.back().second);
    b = F == pts.back().first ? 0 : 1;
  } else {
    size_t k = 1;
    while (pts[k].first < F) ++k;
    const auto& lo = pts[k - 1];
    const auto& hi = pts[k];
    t = hi.first == lo.first ? lo.second : lo.second + (F - lo.first) * (hi.second - lo.second) / (hi.first - lo.first);
  }
  *step_ms = t;
  if (basis) *basis = b;
  return MLORA_OK;
}

mlora_status mlora_shard_jobs_multi(const mlora_problem* problems, int32_t n_problems, const mlora_segment* segs,
                                    int32_t n_segs, int32_t n_ranks, int32_t* rank_of_job, double* load) {
  if (!problems || n_problems < 1 || !segs || !rank_of_job || n_segs < 1 || n_ranks < 1)
    return fail(MLORA_ERR_INVALID, "bad arguments to mlora_shard_jobs");
  // a job's share of one step: per projection, its tokens through the base products plus its
  // three rank-r_i passes over (d_in + d_out)
  double dd = 0.0, ds = 0.0;
  for (int p = 0; p < n_problems; ++p) {
    if (problems[p].d_in < 1 || problems[p].d_out < 1) return fail(MLORA_ERR_INVALID, "bad problem in mlora_shard_jobs");
    dd += static_cast<double>(problems[p].d_in) * problems[p].d_out;
    ds += static_cast<double>(problems[p].d_in) + problems[p].d_out;
  }
  std::vector<std::pair<double, int>> cost(n_segs);
  for (int i = 0; i < n_segs; ++i) {
    if (segs[i].n_tokens < 1 || segs[i].rank < 1) return fail(MLORA_ERR_INVALID, "bad job in mlora_shard_jobs");
    cost[i] = {static_cast<double>(segs[i].n_tokens) * (dd + 3.0 * segs[i].rank * ds), i};
  }
  // longest processing time first onto the least-loaded rank (ties: lowest job index, lowest rank)
  std::stable_sort(cost.begin(), cost.end(), [](const auto& a, const auto& b) { return a.first > b.first; });
  std::vector<double> l(n_ranks, 0.0);
  for (const auto& c : cost) {
    int best = 0;
    for (int r = 1; r < n_ranks; ++r)
      if (l[r] < l[best]) best = r;
    rank_of_job[c.second] = best;
    l[best] += c.first;
  }
  if (load) std::copy(l.begin(), l.end(), load);
  return MLORA_OK;
}

mlora_status mlora_shard_jobs(const mlora_problem* problem, const mlora_segment* segs, int32_t n_segs,
                              int32_t n_ranks, int32_t* rank_of_job, double* load) {
  return mlora_shard_jobs_multi(problem, problem ? 1 : 0, segs, n_segs, n_ranks, rank_of_job, load);
}

const char* mlora_status_string(mlora_status s) {
  switch (s) {
    case MLORA_OK: return "ok";
    case MLORA_ERR_INVALID: return "invalid argument";
    case MLORA_ERR_UNSUPPORTED: return "unsupported";
    case MLORA_ERR_CUDA: return "CUDA error";
    case MLORA_ERR_TIMEOUT: return "device wait timed out";
    case MLORA_ERR_OOM: return "out of memory";
  }
  return "unknown status";
}

const char* mlora_last_error(void) { return g_last_error.c_str(); }

int32_t mlora_version(void) { return 100; }

}  // extern "C"
