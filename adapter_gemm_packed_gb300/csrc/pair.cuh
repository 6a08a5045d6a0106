// Helpers for kernels that run on CTA pairs (cluster of 2, tcgen05 cta_group::2): cluster rank and
// address mapping, pair-wide TMEM allocation, pair MMA and commit, TMA copies whose completion is
// counted on the even CTA's barrier, and the raster of 256-token tile pairs.
#pragma once

#include "common.cuh"

namespace mlora {
namespace pair {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on an mbarrier that
// may live in the peer CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// Same, with an L2 cache policy (see l2_policy_*).
__device__ __forceinline__ void tma_load_2d_pair_hint(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int x,
                                                      int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void umma_pair_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once each) on the barrier at this offset in every CTA of `mask` when all MMAs issued
// so far by this thread have completed.
__device__ __forceinline__ void umma_pair_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(mask)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// Signal a barrier of a CTA of the cluster through the async proxy: a 16-byte bulk copy from
// this CTA's shared memory into `dst_cluster`, completing 16 bytes of transaction count on
// `bar_cluster` (a barrier in the destination CTA).  Unlike a cluster-scope release arrive, the
// issuing thread does not wait for its earlier memory operations to be acknowledged.
__device__ __forceinline__ void bulk_signal_remote(uint32_t dst_cluster, const void* src, uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], 16, [%2];" ::"r"(
                   dst_cluster),
               "r"(smem_u32(src)), "r"(bar_cluster)
               : "memory");
}

// TMA tile store of a box from this CTA's shared memory into global memory (a bulk async-group
// of the issuing thread; the box's swizzle is the tensor map's).  Parts of the box outside the
// tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

// Close the issuing thread's bulk async operations into a group (an empty group if there are none).
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of the issuing thread's most recent bulk groups are still reading their
// shared-memory source (the older ones' sources may be overwritten).
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of the issuing thread's most recent bulk groups are incomplete (their
// writes performed).
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy writes to shared memory before later async-proxy reads of it
// (a TMA store issued after a barrier).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Named barrier `id` over `n` threads (a multiple of 32) that also returns the AND of `pred`
// over them: every participant gets the same decision.
__device__ __forceinline__ int named_bar_and(int id, int n, int pred) {
  int out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(pred), "r"(id), "r"(n)
      : "memory");
  return out;
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Teardown of a CTA pair's main ring.  Every copy into a ring slot, whichever CTA issues it,
// counts on the even CTA's full barrier of that slot, and every issuer fills ring position p only
// after the MMA released position p - S.  So once no thread can issue any more (a cluster barrier
// after all roles have finished), the copies of every position below hi - S have landed, where hi
// is one past the highest position any issuer of either CTA filled.  Each issuer publishes its
// count of filled positions into the even CTA's `ring_hi` (cluster-scope max) before that barrier.
__device__ __forceinline__ void publish_ring_pos(uint32_t* ring_hi, uint32_t filled) {
  const uint32_t addr = mapa_shared(smem_u32(ring_hi), 0);
  asm volatile("red.release.cluster.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(filled) : "memory");
}

// Then the even CTA waits, position by position and bounded, for the last S positions' full
// barriers (position p is slot p % S, phase parity (p / S) & 1; older phases of the same slot have
// completed, so the parity names the right phase).  A position whose copies were not all issued
// never completes: its wait gives up after the timeout, by which time everything issued before
// the barrier has landed, so the remaining positions need no wait.  The final cluster barrier
// keeps the odd CTA's shared memory alive until this drain has finished.
template <int S>
__device__ __forceinline__ void drain_ring(uint64_t* full, uint32_t hi, int* err, unsigned long long timeout_ns) {
  volatile int no_abort = 0;
  for (uint32_t p = hi > S ? hi - S : 0; p < hi; ++p)
    if (!mbar_wait(&full[p % S], (p / S) & 1u, &no_abort, err, DEV_ERR_TIMEOUT_TEARDOWN, timeout_ns)) break;
}

// Raster of the CTA-pair base GEMMs' full tiles.  Items are visited in groups of g.group_m
// tiles along one dimension, sweeping the other: with raster_n == 0 a group is group_m token
// pairs (m fastest) and the group's rows of A stay in L2 while it sweeps every output tile;
// with raster_n == 1 a group is group_m output tiles (n fastest) and its columns of B (the
// weight) stay in L2 while it sweeps every token pair.  The planner picks the order and the
// group size per GEMM from the operands' panel sizes.
__host__ __device__ __forceinline__ void decode_pair(const GemmArgs& g, int item, int& mp, int& n) {
  const int n_pairs = (g.n_mtiles + 1) >> 1;
  const int outer_total = g.raster_n ? n_pairs : g.n_tiles_n;     // swept dimension
  const int inner_total = g.raster_n ? g.n_tiles_n : n_pairs;     // grouped dimension
  const int per_group = g.group_m * outer_total;
  const int group = item / per_group;
  const int first = group * g.group_m;
  const int gsz = inner_total - first < g.group_m ? inner_total - first : g.group_m;
  const int in_group = item - group * per_group;
  const int inner = first + in_group % gsz;
  const int outer = in_group / gsz;
  mp = g.raster_n ? outer : inner;
  n = g.raster_n ? inner : outer;
}


// Item -> (token pair, first output column, width): full tiles in the raster order of
// decode_pair, then the halves of the remaining tiles (two items each).
__host__ __device__ __forceinline__ void decode_item(const GemmArgs& g, int item, int& mp, int& col0, int& width) {
  int n;
  if (item < g.n_full_items) {
    decode_pair(g, item, mp, n);
    col0 = n * BN;
    width = BN;
  } else {
    const int j = item - g.n_full_items;
    decode_pair(g, g.n_full_items + (j >> 1), mp, n);
    col0 = n * BN + (j & 1) * (BN / 2);
    width = BN / 2;
  }
}

}  // namespace pair
}  // namespace mlora
