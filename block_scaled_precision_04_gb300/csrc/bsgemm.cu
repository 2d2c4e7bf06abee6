// bsgemm.cu -- block-scaled (MX) batched GEMM + global Amax for sm_103a.
//
// Operation ("GEMM + Amax (SM100)", section "Equations"):
//   C[m,n,l] = sum_k dec(A[m,k,l]) sf(SFA[m,k/sfv,l]) * dec(B[n,k,l]) sf(SFB[n,k/sfv,l])
//   Amax     = max |C|  (over the values as stored in C's dtype)
// sf(byte) = 2^(byte - 127) for E8M0 scales, the E4M3 value for the NVFP4
// form (E2M1 operands, sfv 16).  A/B are k-major, or (FP8) m-/n-major tiles
// read through the instruction descriptor's transpose bits.  C is fp32,
// fp16 or bf16, or (E2M1 operands) E4M3, E5M2 or packed E2M1.
//
// Kernel design (one persistent CTA per SM, 15 warps; by default two CTAs
// of a cluster form a cta_group::2 pair running 256-row MMAs):
//   warp 0      operand producer: per K stage, the 128 x 128-byte A tile and
//               the B tile (its half in a pair, always whole 128-row boxes)
//               through 3-D tensor maps (128-byte swizzle, out-of-range rows
//               and columns zero-filled).  In a pair both CTAs count their
//               bytes on the leader's stage barrier, which counts copies
//               alone.
//   warp 1      MMA issuer (the leader's, in a pair): once a stage is ready,
//               block-scaled tcgen05.mma (kind::mxf8f6f4 scale_vec::1X for
//               FP8, kind::mxf4nvf4 scale_vec::4X / 2X for packed FP4) into
//               fp32 accumulators in tensor memory; commits free the smem stage
//               and publish a finished accumulator.
//   warps 2..5  scale warps: tcgen05.st of each stage's scale atoms from
//               shared into tensor memory (one warp per lane quarter), then
//               an arrival on the stage's scale barrier, which the MMA tests
//               together with the operand barrier.
//   warps 6..13 epilogue: tcgen05.ld the accumulator (one row per thread),
//               round to C's dtype, keep max |stored value| as an integer max
//               of the float bits, store through a per-warp staging buffer.
//   warp 14     scale producer: each stage's scale atoms in two 4-D tensor
//               copies, on their own barrier, ahead of the operand tiles.
//   The last CTA to finish writes Amax and re-zeroes the workspace slots.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// an error word in the workspace, stops its pipeline, drains in-flight
// copies and MMAs, frees tensor memory and returns.  The drains wait on the
// barriers the copies and MMAs complete on, so they end as soon as those do.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>

#include "bsgemm.h"

namespace {

constexpr int kTileM = 128;
constexpr int kStageKBytes = 128;  // bytes of K per operand row per stage (one swizzle row)
constexpr int kMmaKBytes = 32;     // bytes of K per tcgen05.mma (32 FP8 or 64 FP4 elements)
// Warp roles: 0 operand producer (A/B tiles), 1 MMA issuer, 2-5 scale warps
// (tensor-memory lane quarters 2, 3, 0, 1), 6-13 epilogue (two warps per lane
// quarter), 14 scale producer (tensor copies of the scale atoms).
constexpr int kSfWarp0 = 2;
constexpr int kEpiWarp0 = 6;
constexpr int kEpiWarps = 8;  // (epi_barrier_and counts their 256 threads)
constexpr int kSfProdWarp = kEpiWarp0 + kEpiWarps;
constexpr int kThreads = 32 * (kSfProdWarp + 1);
constexpr int kAtomBytes = 512;    // one scale atom: 128 rows x 4 K-blocks
constexpr int kEpiStageBytes = 2048;  // per epilogue warp: 32 rows x 64 bytes of C
constexpr uint32_t kTmemCols = 512;

// error word bits (workspace word 2); word 3 keeps where the first wait gave up
constexpr uint32_t kErrTimeout = 1u;

enum MmaKind : int { kKindF8F6F4 = 0, kKindF4x4X = 1, kKindF4x2X = 2 };

struct Params {
  int M, N, K, L;
  int tiles_m, tiles_n, num_tiles;
  int tiles_mc;           // groups of cluster_m consecutive M tiles: ceil(tiles_m / cluster_m)
  int num_units;          // scheduling units (one per cluster): full_units + 2 * split tiles
  int full_units;         // units that are whole tiles; the rest are half-width tiles
  int k_bytes;            // bytes per operand row
  int k_stages;           // ceil(k_bytes / 128)
  int t_m, t_n, t_k;      // scale atoms: ceil(M/128), ceil(N/128), ceil(K/(4 sfv))
  int tile_n;
  int stages;
  int c_dtype;            // bsg_dtype
  int c_major;            // 0 = n-major, 1 = m-major
  int a_mn, b_mn;         // 1: A m-major / B n-major (FP8), tiles stored MN-contiguous
  uint32_t idesc;         // instruction descriptor, scale ids zero
  uint32_t idesc_half;    // the same with N = TILE_N / 2 (half-width units)
  uint32_t smem_a, smem_b, smem_sfa, smem_sfb, smem_epi, smem_bar;  // offsets in dynamic smem
  const uint8_t* sfa;
  const uint8_t* sfb;
  void* c;
  float* amax;
  uint32_t* ws;
  unsigned long long wait_limit_ns;
  // tiles left over after the whole waves, each run as two K halves (0: none)
  int ks_tiles;
  int ks_k0;              // first K stage of the second half
  int ks_first;           // index of the first split tile (they follow the whole ones)
  float* part;            // per split tile, K half and CTA rank: 128 x 256 fp32 partial sums
  uint32_t* ks_cnt;       // per split tile and CTA rank: halves claimed, partial sum out
};

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// 4-D tiled copy (scale atoms: 64 x 8-byte words, K atoms, MN atoms, L).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// A pair's second CTA: the box lands in its own shared memory and the bytes
// are counted on the mbarrier at `bar`, a shared::cluster address in the
// pair's leader, so the leader's MMA issuer sees both halves on one barrier.
__device__ __forceinline__ void tma_load_3d_to_leader(uint32_t dst, const CUtensorMap* map, int x,
                                                      int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// cta_group::2 forms: issued by the leader CTA of a pair, acting on both CTAs
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Complete `bytes` of the current phase's transaction count without arriving
// (the drain's stand-in for copies that were never issued).
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// A 32-bit store into the shared memory of another CTA of the cluster.
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Arrive on an mbarrier anywhere in the cluster, releasing this thread's
// earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster_release(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Arrive on an mbarrier anywhere in the cluster (default semantics).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}


__device__ __forceinline__ void tc_mma_pair(int kind, uint32_t d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                            uint32_t accumulate) {
  if (kind == kKindF8F6F4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
  } else if (kind == kKindF4x4X) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
  }
}

__device__ __forceinline__ void tc_mma(int kind, uint32_t d, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                       uint32_t accumulate) {
  if (kind == kKindF8F6F4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
  } else if (kind == kKindF4x4X) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
  }
}

// 32 lanes x 16 consecutive 32-bit columns: thread i gets lane (base + i).
// No wait: follow with tc_wait_ld() before reading r.
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
      "14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 4 consecutive 32-bit columns from registers: thread i writes lane (base + i).
__device__ __forceinline__ void tc_st_32x32b_x4(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


// Shared-memory matrix descriptor, K-major operand tile with 128-byte
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
// K-major tiles: rows of 128 K bytes, 8-row groups 1024 bytes apart (the
// stride byte offset); the leading byte offset is unused.  MN-major tiles:
// rows of 128 MN bytes, one row per K, 8-row (8-K) groups 1024 bytes apart;
// each operand's MN extent per CTA is one 128-byte swizzle span, so the
// leading offset (the step to the next MN span) is never taken -- it is set
// to the same 1024 bytes.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo_bytes = 16) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(lbo_bytes >> 4) << 16;     // leading byte offset
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}


// ------------------------------------------------------------- helpers

// Per-kind constants: scale atoms per 128-byte K stage, MMAs per atom
// column group, and the scale-byte step between those MMAs.
template <int KIND>
struct KindTraits;
template <>
struct KindTraits<kKindF8F6F4> {  // FP8, block 32: one scale byte per K=32 MMA
  static constexpr int kChunks = 1, kMmasPerChunk = 4, kSfIdStep = 1;
};
template <>
struct KindTraits<kKindF4x4X> {  // FP4, block 16: four scale bytes per K=64 MMA
  static constexpr int kChunks = 4, kMmasPerChunk = 1, kSfIdStep = 0;
};
template <>
struct KindTraits<kKindF4x2X> {  // FP4, block 32: two scale bytes per K=64 MMA
  static constexpr int kChunks = 2, kMmasPerChunk = 2, kSfIdStep = 2;
};

struct Tile {
  int l, mt, nt;
  int half;    // -1: the whole tile; 0 / 1: its left / right half (N = TILE_N / 2)
  int ks;      // -1: all of K; else the split tile whose K half kh this unit is
  int kh;
  int kb, ke;  // the unit's K stages [kb, ke)
};

// Unit u (one per cluster) -> (l, group of cluster_m M tiles, N tile); the
// CTA of rank `rank` takes M tile group * cm + rank (past tiles_m: a ghost
// tile whose rows are all masked, kept so the cluster stays in lockstep).
// Units from full_units on split the last tiles in two halves: the schedule's
// final wave is then half-width tiles, so a partly filled last wave costs half
// a tile time instead of a whole one.
//
// K halves instead (ks_tiles = R > 0, G clusters, at least two whole waves):
// the R tiles past the whole waves each run as two units over the first and
// the second half of the K stages, at full width.  The first halves are
// units 0 .. R-1 and the second halves R .. 2R-1: the first units of
// clusters 0 .. 2R-1, whose epilogues exchange the partial sums while whole
// tiles' MMAs run (a half placed after a whole tile left its epilogue too
// little time for that tile's stores, and a half in the last wave put the
// exchange at the end of the launch; both measured slower).  Every cluster
// then carries at most half a tile more than the whole waves, where a
// half-width tail tile (the other split) takes about as long as a whole one:
// its pipeline is bound by the ring's round trip, not the tensor rate.  The
// whole tiles fill the other units in order.
template <bool KS>
__device__ __forceinline__ Tile tile_coords(const Params& p, int u, int cm, int rank) {
  Tile r;
  r.half = -1;
  r.ks = -1;
  r.kh = 0;
  r.kb = 0;
  r.ke = p.k_stages;
  if (KS && p.ks_tiles > 0) {
    const int R = p.ks_tiles;
    if (u < 2 * R) {
      r.ks = u < R ? u : u - R;
      r.kh = u < R ? 0 : 1;
      u = p.ks_first + r.ks;
      if (r.kh) r.kb = p.ks_k0;
      else r.ke = p.ks_k0;
    } else {
      u -= 2 * R;
    }
  } else if (u >= p.full_units) {
    const int hu = u - p.full_units;
    u = p.full_units + (hu >> 1);
    r.half = hu & 1;
  }
  const int per_batch = p.tiles_mc * p.tiles_n;
  r.l = u / per_batch;
  const int rem = u - r.l * per_batch;
  const int mg = rem / p.tiles_n;
  r.nt = rem - mg * p.tiles_n;
  r.mt = mg * cm + rank;
  return r;
}

// try_wait that may suspend the thread for up to `hint_ns` while the phase is open
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Both phases complete (two independent tests in flight at once).
__device__ __forceinline__ bool mbar_test_wait2(uint32_t bar_a, uint32_t bar_b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred pa, pb;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 pa, [%1], %3;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 pb, [%2], %3;\n\t"
      "and.pred pa, pa, pb;\n\t"
      "selp.u32 %0, 1, 0, pa;\n\t}"
      : "=r"(ok)
      : "r"(bar_a), "r"(bar_b), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded slow path of a wait.  Returns false when the pipeline is abandoned.
// Polls with test_wait: warps parked in a blocking try_wait measurably slow
// the MMA issuer sharing their SM.  `sleep_ns` > 0 (warps off the critical
// path: epilogue, scale warps) naps between polls; 0 spins (producers and
// the MMA issuer, whose wake-up latency is on the critical path).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Params& p,
                                       volatile uint32_t* abort_flag, uint32_t where,
                                       uint32_t sleep_ns) {
  const unsigned long long start = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if (sleep_ns) __nanosleep(sleep_ns);
    if (sleep_ns || (i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - start > p.wait_limit_ns) {
        atomicOr(p.ws + 2, kErrTimeout);
        atomicCAS(p.ws + 3, 0u, where);
        *abort_flag = 1u;
        return false;
      }
    }
  }
}

// AND of `v` over the 256 threads of the 8 epilogue warps, at named barrier 1
// (every epilogue thread must arrive, with no other thread using the id).
__device__ __forceinline__ uint32_t epi_barrier_and(uint32_t v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "barrier.cta.red.and.pred po, 1, 256, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(v)
      : "memory");
  return r;
}

// The K-half hand-off counters in global memory: an acquire load and an
// acq_rel add at GPU scope.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* a) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* a, uint32_t x) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(x)
               : "memory");
  return old;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* a, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// Bounded wait for a flag in global memory another CTA sets (release) once
// work it has already begun is done.  Returns false when the pipeline is
// abandoned, as wait_slow does.
__device__ __noinline__ bool wait_flag_gpu(const uint32_t* f, const Params& p,
                                           volatile uint32_t* abort_flag, uint32_t where) {
  const unsigned long long start = globaltimer();
  while (ld_acquire_gpu(f) == 0u) {
    __nanosleep(64);
    if (*abort_flag) return false;
    if (globaltimer() - start > p.wait_limit_ns) {
      atomicOr(p.ws + 2, kErrTimeout);
      atomicCAS(p.ws + 3, 0u, where);
      *abort_flag = 1u;
      return false;
    }
  }
  return true;
}

// 16 fp32 words of a K-half partial sum from L2: four 16-byte pieces 512
// bytes apart.  One statement, so that the pieces of one chunk are in flight
// together and the next chunk's are not hoisted above this one's adds.
__device__ __forceinline__ void ld_part16(const float4* a, uint32_t (&x)[16]) {
  asm volatile(
      "ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%16];\n\t"
      "ld.global.cg.v4.u32 {%4, %5, %6, %7}, [%16+512];\n\t"
      "ld.global.cg.v4.u32 {%8, %9, %10, %11}, [%16+1024];\n\t"
      "ld.global.cg.v4.u32 {%12, %13, %14, %15}, [%16+1536];"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]),
        "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]),
        "=r"(x[14]), "=r"(x[15])
      : "l"(a)
      : "memory");
}

// Named barrier `id` over `count` threads (whole warps).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("barrier.cta.sync.aligned %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Fast path inline: one test_wait; the bounded loop only when the phase is open.
#define BSG_WAIT(bar, parity, site) \
  (mbar_test_wait((bar), (parity)) || wait_slow((bar), (parity), p, abort_flag, (site), 0u))
#define BSG_WAIT_SLEEP(bar, parity, site) \
  (mbar_test_wait((bar), (parity)) || wait_slow((bar), (parity), p, abort_flag, (site), 128u))

__device__ __forceinline__ uint32_t abs_bits_f32(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// Low-precision C: two fp32 values -> two codes, round to nearest even,
// saturating (`lo` in the low byte / nibble).  E2M1 has no NaN: a NaN is
// stored as +0.
__device__ __forceinline__ uint32_t cvt2_e4m3(float lo, float hi) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
  return h;
}
__device__ __forceinline__ uint32_t cvt2_e5m2(float lo, float hi) {
  uint16_t h;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
  return h;
}
__device__ __forceinline__ uint32_t cvt2_e2m1(float lo, float hi) {
  uint32_t r;
  lo = lo != lo ? 0.0f : lo;
  hi = hi != hi ? 0.0f : hi;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// |value| of a low-precision code (sign ignored) as an fp32, from the
// format's fields: E4M3 (bias 7, S.1111.111 NaN), E5M2 (bias 15, IEEE-like
// infinity / NaN), E2M1 (bias 1, no specials).
__device__ __forceinline__ float decode_mag(uint32_t code, int c_dtype) {
  if (c_dtype == BSG_E4M3) {
    const uint32_t e = (code >> 3) & 15u, m = code & 7u;
    if (e == 15u && m == 7u) return __uint_as_float(0x7FC00000u);
    if (e == 0u) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));
  }
  if (c_dtype == BSG_E5M2) {
    const uint32_t e = (code >> 2) & 31u, m = code & 3u;
    if (e == 31u) return __uint_as_float(m ? 0x7FC00000u : 0x7F800000u);
    if (e == 0u) return static_cast<float>(m) * 1.52587890625e-05f;  // m * 2^-16
    return __uint_as_float(((e + 112u) << 23) | (m << 21));
  }
  const uint32_t e = (code >> 1) & 3u, m = code & 1u;
  if (e == 0u) return 0.5f * static_cast<float>(m);
  return __uint_as_float(((e + 126u) << 23) | (m << 22));
}

// A warp's 32 rows of W 32-bit words (row t in lane t's v[0..W)) to global
// memory, row-major with a pitch of `pitch` bytes from `g` (row 0, word 0),
// through the warp's 2 KB staging buffer `stg`.  Each store instruction then
// writes W/4 lanes x 16 contiguous bytes per row (8 rows x 64 bytes for
// W = 16) instead of 32 scattered 16-byte pieces.  The 16-byte pieces of a
// row sit XOR-swizzled by (row / 2) % 4, which keeps both the row-per-lane
// writes and the piece-per-lane reads free of bank conflicts.  Rows from
// `rows_valid` and bytes from `bytes_valid` (multiples of 16) on are not
// written.
template <int W>
__device__ __forceinline__ void store_rows_coalesced(uint8_t* stg, const uint32_t* v, int lane, char* g,
                                                     size_t pitch, int rows_valid, int bytes_valid) {
  static_assert(W == 8 || W == 16, "a staged row chunk is 32 or 64 bytes");
  constexpr int L = W / 4;    // lanes (16-byte pieces) per row
  constexpr int RP = 32 / L;  // rows per store instruction
  __syncwarp();               // the previous chunk's reads are done
#pragma unroll
  for (int pc = 0; pc < L; ++pc)
    *reinterpret_cast<uint4*>(stg + lane * 64 + ((pc ^ ((lane >> 1) & 3)) * 16)) =
        make_uint4(v[4 * pc], v[4 * pc + 1], v[4 * pc + 2], v[4 * pc + 3]);
  __syncwarp();
#pragma unroll
  for (int k = 0; k < L; ++k) {
    const int r = lane / L + RP * k, pc = lane % L;
    const uint4 x = *reinterpret_cast<const uint4*>(stg + r * 64 + ((pc ^ ((r >> 1) & 3)) * 16));
    if (r < rows_valid && pc * 16 < bytes_valid)
      *reinterpret_cast<uint4*>(g + static_cast<size_t>(r) * pitch + pc * 16) = x;
  }
}

// Bounded wait for the drains at exit (no abort flag: always runs).  It
// waits for this CTA's own copies and MMAs, which finish by themselves, so
// its limit, counted from `start` (one deadline for a whole drain), never
// drops below 200 ms even when the pipeline waits use a shorter one.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const Params& p,
                                           uint32_t where, unsigned long long start) {
  const unsigned long long limit =
      p.wait_limit_ns > 200000000ull ? p.wait_limit_ns : 200000000ull;
  while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (globaltimer() - start > limit) {
      atomicOr(p.ws + 2, kErrTimeout);
      atomicCAS(p.ws + 3, 0u, where);
      break;
    }
  }
}

// --------------------------------------------------------------- kernel

// LOWC: the epilogue writes low-precision C (E4M3, E5M2 or packed E2M1; FP4
// operands only); a kernel of its own, since that path's registers would
// otherwise spill in every FP4 kernel.
template <int KIND, int TILE_N, int NUM_ACC, int CM, int PAIR, int KSL, int LOWC, int KSPL>
__global__ void __launch_bounds__(kThreads, 1)
    bsg_gemm_amax_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_bh,
                         const __grid_constant__ CUtensorMap tmap_sfa,
                         const __grid_constant__ CUtensorMap tmap_sfb, const __grid_constant__ Params p) {
  using KT = KindTraits<KIND>;
  // 128-row scale groups of B the MMA reads (tile rows 128g .. 128g+127 at
  // columns +4g); a tile width that is not a multiple of 128 (224) starts at
  // any multiple of 32 inside a scale atom, so its scales span one atom more
  constexpr int G = (TILE_N + 127) / 128;
  constexpr bool kAlignedN = TILE_N % 128 == 0;
  constexpr int kSfbAtoms = kAlignedN ? G : G + 1;  // B scale atoms per chunk in smem
  // a stage holds KSL 128-byte K slices (each its own 128-byte swizzle block)
  constexpr int kSB = kStageKBytes * KSL;                // K bytes per stage
  constexpr int kCps = KT::kChunks * KSL;                // scale atoms along K per stage
  constexpr uint32_t kASlice = kTileM * kStageKBytes;
  constexpr uint32_t kAStage = kASlice * KSL;            // smem bytes per stage
  // PAIR: a 2-CTA pair runs 256 x TILE_N MMAs (cta_group::2); each CTA holds
  // its 128 rows of A and half (TILE_N/2 rows) of the B tile
  static_assert((CM == 1 && !PAIR) || (CM == 2 && PAIR), "a CTA alone or a cta_group::2 pair");
  constexpr int kBRows = PAIR ? TILE_N / 2 : TILE_N;
  // B is loaded in boxes of whole 128-row groups: a 112-row box (a 224-wide
  // pair's half) streams markedly slower through the TMA unit, so the half
  // is loaded as 128 rows and the MMA reads the first 112
  constexpr int kBLoadRows = (kBRows + 127) / 128 * 128;
  constexpr uint32_t kBSlice = kBLoadRows * kStageKBytes;
  constexpr uint32_t kBStage = kBSlice * KSL;
  constexpr uint32_t kSfaStage = kCps * kAtomBytes;
  constexpr uint32_t kSfbStage = kCps * kAtomBytes * kSfbAtoms;
  // scale columns follow the accumulators, one set per smem stage, so that a
  // stage's tcgen05.st never rewrites columns an in-flight MMA still reads
  constexpr uint32_t kSfCols = 4 * kCps * (1 + G);
  // FP8 256-wide tiles with one accumulator: consecutive units of a CTA
  // alternate between two accumulator regions of tensor memory that share
  // kOvlCols columns -- [kOvlCols, kOvlCols + 256) and [256, 512), the scale
  // sets below them -- so the next unit's MMAs wait only until the epilogue
  // has drained the shared columns, not the whole accumulator
  constexpr bool kOvl = KIND == kKindF8F6F4 && TILE_N == 256 && NUM_ACC == 1;
  constexpr uint32_t kOvlCols = 80;                       // 5 chunks of 16 columns
  constexpr int kPartF4 = kTileM * TILE_N / 4;            // float4 per K-half partial sum buffer
  // the instantiation that runs K halves of the leftover tiles (launched
  // only when a run uses them: the code they need, compiled into every
  // launch, slowed the ordinary one)
  constexpr bool kKs = KSPL != 0 && kOvl;
  constexpr int kRegions = kOvl ? 2 : NUM_ACC;            // accumulator hand-off slots
  constexpr uint32_t kSfCol0 = kOvl ? 0u : NUM_ACC * TILE_N;
  static_assert(!kOvl || 2 * TILE_N <= kTmemCols, "regions fit");
  // tensor-memory column of accumulator slot r
  auto acc_col = [](int r) -> uint32_t {
    return kOvl ? (r ? kTmemCols - TILE_N : kOvlCols) : static_cast<uint32_t>(r) * TILE_N;
  };
  constexpr int kMmasPerStage = kSB / kMmaKBytes;
  constexpr int kMmasPerSlice = kStageKBytes / kMmaKBytes;
  // both CTAs of a pair: the targets of the leader's commit arrivals
  constexpr uint16_t kMask = static_cast<uint16_t>((1u << CM) - 1u);
  // half-width units (the split last wave) exist for 256-wide pairs only:
  // each CTA then loads 64 rows of B (the tmap_bh box) and the MMA runs N = 128
  constexpr bool kHalves = PAIR && TILE_N == 256;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // align the dynamic window to 1024 bytes (128-byte swizzle atoms)
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  const int crank = CM > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int unit0 = CM > 1 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int unit_step = CM > 1 ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);

  const uint32_t bar0 = base + p.smem_bar;
  // per stage:
  //   full  the stage's A/B bytes have landed -- of both CTAs of a pair,
  //         counted in the leader (the leader's expect_tx, both CTAs' copies)
  //   empty the stage is free (the MMA commit; in a pair, in both CTAs)
  //   sff   this CTA's scale bytes have landed (issued first, off the A/B path)
  //   sfr   every scale warp has put the stage's scales in tensor memory (in
  //         the leader; four per CTA)
  //   pd    (second CTA of a pair, at the exit drain) the leader has seen the
  //         stage's bytes land
  // The MMA waits sfr and full.  full counts copies alone, so a producer's
  // exit drain can wait on it for the copies it issued, whatever the rest
  // of the pipeline did after an abort.
  const uint32_t full0 = bar0, empty0 = bar0 + 8u * S, sff0 = bar0 + 16u * S;
  const uint32_t sfr0 = bar0 + 24u * S, pd0 = bar0 + 32u * S;
  // per accumulator slot: accf (accumulator full), acce (fully drained),
  // acco (its columns shared with the other region drained; kOvl only)
  const uint32_t accf0 = bar0 + 40u * S, acce0 = accf0 + 8u * kRegions;
  const uint32_t acco0 = acce0 + 8u * kRegions;
  const uint32_t drain_bar = acco0 + 8u * kRegions;
  const uint32_t pinfo_bar = drain_bar + 8u;  // the second CTA's drain record is in
  uint32_t* const misc =
      reinterpret_cast<uint32_t*>(smem + p.smem_bar + 40u * S + 24u * kRegions + 16u);
  uint32_t* const tmem_holder = misc + 0;
  volatile uint32_t* const abort_flag = misc + 1;
  uint32_t* const cta_amax = misc + 2;
  // the operand producer's record for the exit drain: per stage the bytes it
  // expects (this CTA's share), and (in the leader) the second CTA's record:
  // its armed-stage mask, their parities and per-stage bytes
  uint32_t* const stage_bytes = misc + 4;         // [8]
  uint32_t* const peer_rec = misc + 12;           // [2 + 8]

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);                // the leader's expect_tx
      mbar_init(sfr0 + 8u * s, PAIR ? 8 : 4);      // the scale warps of both CTAs
      mbar_init(pd0 + 8u * s, 1);
      // freed by the MMA commit (in a pair, the leader's commit arrives in
      // both CTAs)
      mbar_init(empty0 + 8u * s, 1);
      mbar_init(sff0 + 8u * s, 1);
    }
    for (int b = 0; b < kRegions; ++b) {
      mbar_init(accf0 + 8u * b, 1);
      mbar_init(acce0 + 8u * b, PAIR ? 2 * kEpiWarps : kEpiWarps);  // one per epilogue warp
      mbar_init(acco0 + 8u * b, PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    mbar_init(pinfo_bar, 1);
    *abort_flag = 0u;
    *cta_amax = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  // The setup's cluster barrier, split: every warp arrives here (thread 0
  // after its barrier inits, which the arrival releases) and waits after the
  // CTA barrier, so that the barrier's latency overlaps the tensor-memory
  // allocation.  The peer's allocation is still ordered before the leader's
  // first MMA: that waits for the peer's scale warps, which start after it.
  if (CM > 1) {
    __syncwarp();
    cluster_arrive();
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
  }
  if (warp == kSfProdWarp && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_sfa)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_sfb)) : "memory");
  }
  if (warp == 1) {
    if (PAIR) {  // one warp of each CTA of the pair allocates collectively
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_holder)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_holder)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CM > 1) cluster_wait();  // the peer's barriers initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // this warp has arrived on the final cluster barrier (the epilogue arrives
  // as soon as its last accumulator release is out, so that the barrier's
  // release does not wait for its last stores)
  bool cl_arrived = false;

  if (warp == 0 || warp == kSfProdWarp) {
    // ----------------------------------------------------- producers
    // warp 0 issues the operand tiles (first thing once a stage frees);
    // warp kSfProdWarp issues the stage's small scale copies on their own
    // barrier.  Both wait on the same stage-free barrier.
    const bool scales = warp == kSfProdWarp;
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // stages with a load issued (for the drain)
      uint32_t armed_parity = 0;
      bool ok = true;
      const uint32_t a_dst0 = base + p.smem_a, b_dst0 = base + p.smem_b;
      const uint32_t sfa_dst0 = base + p.smem_sfa, sfb_dst0 = base + p.smem_sfb;
      const uint32_t bar_base = scales ? sff0 : full0;
      const bool a_mn = KIND == kKindF8F6F4 && p.a_mn, b_mn = KIND == kKindF8F6F4 && p.b_mn;
      for (int u = unit0; u < p.num_units && ok; u += unit_step) {
        const Tile tc = tile_coords<kKs>(p, u, CM, crank);
        const bool hu = kHalves && tc.half >= 0;
        const int m0 = tc.mt * kTileM;
        const int n0 = tc.nt * TILE_N + (hu ? tc.half * (TILE_N / 2) : 0);
        const int atom0 = n0 / 128;  // first scale atom of B covering this unit
        // B rows per CTA of this unit, their tensor map and the stage's bytes
        const int brows = hu ? kBRows / 2 : kBRows;
        const CUtensorMap* const bmap = hu ? &tmap_bh : &tmap_b;
        const uint32_t b_stage_bytes = hu ? kBStage / 2 : kBStage;
        for (int ks = tc.kb; ks < tc.ke; ++ks) {
          if (!BSG_WAIT(empty0 + 8u * stage, phase ^ 1u, scales ? 12 : 1)) { ok = false; break; }
          const uint32_t bar = bar_base + 8u * stage;
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (scales) {
            // the stage's scale atoms in two tensor copies (the small copies
            // share the TMA unit with the operand tiles, so fewer is faster):
            // atoms past the tensor's end (a ghost M tile, N or K tails)
            // arrive zero-filled and are never read for a stored element
            mbar_arrive_expect_tx(bar, kSfaStage + kSfbStage);
            tma_load_4d(sfa_dst0 + stage * kSfaStage, &tmap_sfa, 0, ks * kCps, tc.mt, tc.l, bar);
            tma_load_4d(sfb_dst0 + stage * kSfbStage, &tmap_sfb, 0, ks * kCps, atom0, tc.l, bar);
          } else if (PAIR && crank != 0) {
            // the second CTA of a pair: its halves are counted in the leader
            stage_bytes[stage] = kAStage + b_stage_bytes;
            const uint32_t lbar = mapa_shared(bar, 0);
#pragma unroll
            for (int sl = 0; sl < KSL; ++sl) {
              const int kx = ks * kSB + sl * kStageKBytes;
              const int nb = n0 + brows;
              // a k-major box is (K bytes, rows); an MN-major one (MN, K rows)
              tma_load_3d_to_leader(a_dst0 + stage * kAStage + sl * kASlice, &tmap_a,
                                    a_mn ? m0 : kx, a_mn ? kx : m0, tc.l, lbar);
              tma_load_3d_to_leader(b_dst0 + stage * kBStage + sl * kBSlice, bmap,
                                    b_mn ? nb : kx, b_mn ? kx : nb, tc.l, lbar);
            }
          } else {
            // a pair's leader expects the bytes of both CTAs
            stage_bytes[stage] = kAStage + b_stage_bytes;
            mbar_arrive_expect_tx(bar, (PAIR ? 2u : 1u) * (kAStage + b_stage_bytes));
#pragma unroll
            for (int sl = 0; sl < KSL; ++sl) {
              const int kx = ks * kSB + sl * kStageKBytes;
              tma_load_3d(a_dst0 + stage * kAStage + sl * kASlice, &tmap_a, a_mn ? m0 : kx,
                          a_mn ? kx : m0, tc.l, bar);
              tma_load_3d(b_dst0 + stage * kBStage + sl * kBSlice, bmap, b_mn ? n0 : kx,
                          b_mn ? kx : n0, tc.l, bar);
            }
          }
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      // drain: every issued load must have landed before the CTA may exit,
      // observed on the barriers the copies complete on (the rest of the
      // pipeline may have given up after an abort).
      const unsigned long long t_drain = globaltimer();
      if (scales || !PAIR) {
        // the scale copies on this CTA's sff; a lone CTA's operand copies on
        // its full, which counts copies alone
        for (int s = 0; s < S; ++s)
          if (armed & (1u << s))
            drain_wait((scales ? sff0 : full0) + 8u * s, (armed_parity >> s) & 1u, p,
                       scales ? 13u : 10u, t_drain);
      } else if (crank != 0) {
        // second CTA of a pair: its copies complete on the leader's full.
        // Hand the leader this CTA's record, then wait for its word, per
        // stage, that the stage's bytes have landed.
        const uint32_t lrec = mapa_shared(smem_u32(peer_rec), 0);
        st_cluster_u32(lrec, armed);
        st_cluster_u32(lrec + 4u, armed_parity);
        for (int s = 0; s < S; ++s) st_cluster_u32(lrec + 8u + 4u * s, stage_bytes[s]);
        mbar_arrive_cluster_release(mapa_shared(pinfo_bar, 0));
        for (int s = 0; s < S; ++s)
          if (armed & (1u << s)) drain_wait(pd0 + 8u * s, 0u, p, 17u, t_drain);
      } else {
        // the leader: its full counts both CTAs' copies.  With the second
        // CTA's record (if it arrives), a stage only one of the two issued
        // after an abort is completed by hand: the share that will never
        // come off the count, or the expect_tx that was never made.
        drain_wait(pinfo_bar, 0u, p, 18u, t_drain);
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        // without the record (its wait gave up), assume the second CTA
        // issued what this one did
        const bool rec = mbar_test_wait(pinfo_bar, 0u);
        const uint32_t pm = rec ? peer_rec[0] : armed, pp = rec ? peer_rec[1] : armed_parity;
        const uint32_t* const precs = rec ? peer_rec + 2 : stage_bytes;
        for (int s = 0; s < S; ++s) {
          const bool mine = (armed >> s) & 1u, theirs = (pm >> s) & 1u;
          if (!mine && !theirs) continue;
          const uint32_t bar = full0 + 8u * s;
          const uint32_t mp = (armed_parity >> s) & 1u, tp = (pp >> s) & 1u;
          // the phase both issued, or the newer of two (the older one is
          // complete: a newer arming needs the older phase consumed)
          uint32_t parity = mine ? mp : tp;
          if (mine && theirs && mp != tp) {
            if (mbar_test_wait(bar, mp)) {
              parity = tp;  // ours is the older: the second CTA's phase lacks our expect_tx
              mbar_arrive_expect_tx(bar, precs[s]);
            } else {
              mbar_complete_tx(bar, stage_bytes[s]);  // ours lacks the second CTA's bytes
            }
          } else if (mine && !theirs) {
            mbar_complete_tx(bar, stage_bytes[s]);
          } else if (!mine && theirs) {
            mbar_arrive_expect_tx(bar, precs[s]);
          }
          drain_wait(bar, parity, p, 10u, t_drain);
          if (theirs) mbar_arrive_cluster(mapa_shared(pd0 + 8u * s, 1));
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    // (in a CTA pair only the leader issues, for both CTAs).  The whole warp
    // walks the loop, so the descriptors and addresses stay warp-uniform, and
    // one elected lane issues the MMAs and commits: issuing from a
    // single-lane branch measured ~120 cycles per tcgen05.mma against ~63
    // this way, which left the tensor pipe idle between stages.
    if (!PAIR || crank == 0) {
      const bool elected = elect_one();
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // descriptors of stage 0; a stage or MMA step adds a constant to the
      // 16-byte-granular start address in the low bits
      const bool a_mn = KIND == kKindF8F6F4 && p.a_mn, b_mn = KIND == kKindF8F6F4 && p.b_mn;
      const uint64_t adesc0 = desc_sw128(base + p.smem_a, a_mn ? 1024u : 16u);
      const uint64_t bdesc0 = desc_sw128(base + p.smem_b, b_mn ? 1024u : 16u);
      // start-address step (16-byte units) of one MMA's K: 32 bytes along a
      // k-major row, or 32 rows of 128 bytes in an MN-major tile
      const uint32_t a_kstep = a_mn ? (kMmaKBytes * 128) >> 4 : kMmaKBytes >> 4;
      const uint32_t b_kstep = b_mn ? (kMmaKBytes * 128) >> 4 : kMmaKBytes >> 4;
      const uint32_t sf_t0 = tmem + kSfCol0;
      const uint32_t idesc = p.idesc;
      auto mma_issue = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t sa,
                           uint32_t sb, uint32_t accumulate) {
        if (PAIR) tc_mma_pair(KIND, d, a, b, id, sa, sb, accumulate);
        else tc_mma(KIND, d, a, b, id, sa, sb, accumulate);
      };
      // running addresses of the current stage
      uint64_t ad = adesc0, bd = bdesc0;
      uint32_t sfa_t = sf_t0;
      const int last = p.k_stages - 1;
      int last_nmma = (p.k_bytes - last * kSB + kMmaKBytes - 1) / kMmaKBytes;
      if (last_nmma > kMmasPerStage) last_nmma = kMmasPerStage;
      uint32_t ovp0 = 0, ovp1 = 0;  // parity of the next shared-column release per slot
      bool first_unit = true;
      for (int u = unit0; u < p.num_units && ok; u += unit_step) {
        if (!BSG_WAIT(acce0 + 8u * acc, acc_phase ^ 1u, 2)) { ok = false; break; }
        if (kOvl && !first_unit) {
          // the previous unit (in the other slot) has drained the columns the
          // two regions share
          const int other = acc ^ 1;
          if (!BSG_WAIT(acco0 + 8u * other, other ? ovp1 : ovp0, 14)) { ok = false; break; }
          if (other) ovp1 ^= 1u;
          else ovp0 ^= 1u;
        }
        first_unit = false;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc_col(acc);
        // a half-width unit runs N = TILE_N / 2 from the first half of each
        // CTA's B rows into the first TILE_N / 2 accumulator columns
        const uint32_t id_u = kHalves && u >= p.full_units ? p.idesc_half : idesc;
        // the unit's K stages (a K half of a split tile: part of them)
        const Tile tc = tile_coords<kKs>(p, u, CM, crank);
        const int kb = tc.kb;
        for (int ks = kb; ks < tc.ke; ++ks) {
          // this stage's scales in tensor memory and its operands in smem:
          // both barriers tested at once on the fast path
          if (!(mbar_test_wait2(sfr0 + 8u * stage, full0 + 8u * stage, phase) ||
                (BSG_WAIT(sfr0 + 8u * stage, phase, 16) && BSG_WAIT(full0 + 8u * stage, phase, 3)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfb_t = sfa_t + 4 * kCps;
          const int nm = ks == last ? last_nmma : kMmasPerStage;
          if (elected) {
#pragma unroll
          for (int j = 0; j < kMmasPerStage; ++j) {
            if (j < nm) {
              const int c = j / KT::kMmasPerChunk;
              const uint32_t sf_id = static_cast<uint32_t>((j % KT::kMmasPerChunk) * KT::kSfIdStep);
              const int sl = j / kMmasPerSlice, jj = j % kMmasPerSlice;
              mma_issue(d_tmem, ad + ((sl * kASlice) >> 4) + jj * a_kstep,
                        bd + ((sl * kBSlice) >> 4) + jj * b_kstep,
                        id_u | (sf_id << 29) | (sf_id << 4), sfa_t + 4 * c, sfb_t + 4 * G * c,
                        (j != 0 || ks != kb) ? 1u : 0u);
            }
          }
          // frees the smem stage (in both CTAs of a pair) once these MMAs
          // finish; issued at once, since the ring is latency-bound and every
          // cycle of delay here delays the stage's refill
          if (PAIR) tc_commit_pair_mc(empty0 + 8u * stage, kMask);
          else tc_commit(empty0 + 8u * stage);
          }
          __syncwarp();
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
            ad = adesc0;
            bd = bdesc0;
            sfa_t = sf_t0;
          } else {
            ad += kAStage >> 4;
            bd += kBStage >> 4;
            sfa_t += kSfCols;
          }
        }
        if (!ok) break;
        // accumulator ready for the epilogue (of both CTAs of a pair)
        if (elected) {
          if (PAIR) tc_commit_pair_mc(accf0 + 8u * acc, kMask);
          else tc_commit(accf0 + 8u * acc);
        }
        __syncwarp();
        if (++acc == kRegions) { acc = 0; acc_phase ^= 1u; }
      }
      // drain: all MMAs issued by this warp complete before exit
      if (elected) {
        if (PAIR) tc_commit_pair(drain_bar);
        else tc_commit(drain_bar);
        drain_wait(drain_bar, 0, p, 11u, globaltimer());
      }
      __syncwarp();
    }
  } else if (warp >= kSfWarp0 && warp < kSfWarp0 + 4) {
    // --------------------------------------------------------- scale warps
    // Per stage, once its bytes have landed, lane i of warp q = w % 4 moves
    // row i of every scale atom of the stage (16 bytes: rows i, 32+i, 64+i,
    // 96+i of a 128-row group, 4 K-blocks each) into tensor-memory lane
    // 32q + i of the stage's scale columns, which gives each lane quarter the
    // atom layout the block-scaled MMA reads.  Scale copies thus never sit in
    // the MMA thread's issue stream.
    const int q = warp & 3;
    int stage = 0;
    uint32_t phase = 0;
    const uint32_t lane_off = static_cast<uint32_t>(lane) * 16u;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16) + kSfCol0;
    bool ok = true;
    for (int u = unit0; u < p.num_units && ok; u += unit_step) {
      // row offset of the tile's first B row inside its first scale atom
      const Tile tc = tile_coords<kKs>(p, u, CM, crank);
      const int n_off = (tc.nt * TILE_N) % 128;
      for (int ks = tc.kb; ks < tc.ke; ++ks) {
        // one lane sleeps on the barrier (the scale bytes are issued ahead of
        // the operand tiles, so there is slack; a polling warp would steal
        // issue slots from the MMA warp, which shares a sub-partition with
        // the quarter-1 scale warp); then every lane observes the completed
        // phase itself before reading the bytes
        int landed = 1;
        if (lane == 0) landed = BSG_WAIT_SLEEP(sff0 + 8u * stage, phase, 5) ? 1 : 0;
        if (!__shfl_sync(0xFFFFFFFFu, landed, 0)) { ok = false; break; }
        mbar_test_wait(sff0 + 8u * stage, phase);
        const uint8_t* sa = smem + p.smem_sfa + stage * kSfaStage + lane_off;
        const uint8_t* sb = smem + p.smem_sfb + stage * kSfbStage + lane_off;
        const uint32_t tcol = t_row + stage * kSfCols;
#pragma unroll
        for (int c = 0; c < kCps; ++c) {
          tc_st_32x32b_x4(tcol + 4 * c, *reinterpret_cast<const uint4*>(sa + c * kAtomBytes));
          if (kAlignedN) {
#pragma unroll
            for (int g = 0; g < G; ++g)
              tc_st_32x32b_x4(tcol + 4 * kCps + 4 * (c * G + g),
                              *reinterpret_cast<const uint4*>(sb + g * kSfaStage + c * kAtomBytes));
          } else {
            // gather: tile row 128g + 32m1 + lane is row lane of the atom
            // holding B row n0 + that row (n_off is a multiple of 32)
#pragma unroll
            for (int g = 0; g < G; ++g) {
              uint32_t w[4];
#pragma unroll
              for (int m1 = 0; m1 < 4; ++m1) {
                const int t = 128 * g + 32 * m1;
                const int rr = n_off + t;
                w[m1] = t < TILE_N ? *reinterpret_cast<const uint32_t*>(
                                         sb + (rr >> 7) * kSfaStage + c * kAtomBytes + ((rr >> 5) & 3) * 4)
                                   : 0x7F7F7F7Fu;  // rows past the tile: scale 1
              }
              tc_st_32x32b_x4(tcol + 4 * kCps + 4 * (c * G + g), make_uint4(w[0], w[1], w[2], w[3]));
            }
          }
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        // one of the stage's arrivals (on the leader's barrier in a pair)
        if (lane == 0) {
          if (PAIR) mbar_arrive_cluster(mapa_shared(sfr0 + 8u * stage, 0));
          else mbar_arrive(sfr0 + 8u * stage);
        }
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    // Warp w reads lane quarter q = w % 4 and column half h of the tile (one
    // row per thread, TILE_N/2 columns).  16-bit C: each 16-column chunk is
    // rounded and packed as it leaves tensor memory, the accumulator is
    // released after the last chunk, and the stores overlap the next tile's
    // MMAs.  fp32 C: two passes of TILE_N/4 columns, released after the
    // second pass's loads.
    constexpr int kCols = TILE_N / 2;  // columns of this warp in a whole tile
    constexpr int kRnd = 4;            // chunks per round of tensor-memory loads
    const int q = warp & 3;
    const int h = (warp - kEpiWarp0) >> 2;
    uint8_t* const stg = smem + p.smem_epi + (warp - kEpiWarp0) * kEpiStageBytes;
    // max |stored value|, kept per C dtype and turned into fp32 bits at the
    // end: fp32 C -> the fp32 bits; 16-bit C -> two packed 16-bit magnitudes
    // (they order like their values, so an unsigned SIMD max finds the
    // largest); FP8 / E2M1 C -> the largest stored |C| before rounding
    uint32_t vmax = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = unit0; u < p.num_units; u += unit_step) {
      const Tile tc = tile_coords<kKs>(p, u, CM, crank);
      // one lane of one warp spins on the accumulator; the 8 epilogue warps
      // take its verdict at a named barrier, which also wakes them at once
      // (napping warps added up to a nap's length to every hand-off)
      uint32_t ready = 1;
      // a K half: the same lane claims the split tile before the wait, so
      // that the claim's round trip stays off the accumulator hand-off
      uint32_t ks_first = 1;
      if (warp == kEpiWarp0 && lane == 0) {
        if constexpr (kKs) {
          if (tc.ks >= 0) ks_first = atom_add_acq_rel_gpu(p.ks_cnt + 4 * tc.ks + 2 * crank, 1u) == 0u;
        }
        ready = BSG_WAIT(accf0 + 8u * acc, acc_phase, 4) ? 1u : 0u;
      }
      if (!epi_barrier_and(ready)) break;
      tc_fence_after();
      // a half-width unit (N = TILE_N / 2 in the first accumulator columns)
      // gives each warp half as many columns
      const bool hu = kHalves && tc.half >= 0;
      const int ucol0 = tc.nt * TILE_N + (hu ? tc.half * (TILE_N / 2) : 0);
      const int slot = acc;  // accumulator slot of this unit
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc_col(slot);
      const int row = tc.mt * kTileM + q * 32 + lane;
      const bool row_ok = row < p.M;
      const size_t batch_off = static_cast<size_t>(tc.l) * p.M * p.N;
      const uint32_t release_bar = acce0 + 8u * slot;
      const uint32_t shared_bar = acco0 + 8u * slot;
      const bool last_unit = u + unit_step >= p.num_units;
      if (++acc == kRegions) { acc = 0; acc_phase ^= 1u; }
      // this warp is done reading the accumulator (release) or the columns
      // its region shares with the other (release_shared, kOvl only)
      auto arrive_on = [&](uint32_t bar) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR) mbar_arrive_cluster(mapa_shared(bar, 0));
          else mbar_arrive(bar);
        }
      };
      auto release = [&]() {
        arrive_on(release_bar);
        if (CM > 1 && last_unit) {  // no remote access follows in this warp
          __syncwarp();             // (lane 0 alone made the arrival)
          cluster_arrive();
          cl_arrived = true;
        }
      };
      auto release_shared = [&]() { arrive_on(shared_bar); };
      // K halves of a split tile (kOvl kernels).  src 0: a unit over all of K;
      // 2: this half claimed the tile first and publishes its partial sum;
      // 1: the other half claimed first: this half parks its own partial sum
      // too (freeing its tensor memory at once, as the claimant does), waits
      // for the claimant's, and stores C from the two.  fp32 addition is
      // commutative, so C does not depend on which half is which.
      int src = 0;
      // float4 offset in p.part of this CTA rank's buffer of K half kh
      auto part_of = [&](int kh) { return (4 * tc.ks + 2 * kh + crank) * kPartF4; };
      // a partial sum buffer holds, per 16-column chunk ch of the unit, lane
      // quarter q and 16-byte piece v, the 32 lanes' pieces in 512 contiguous
      // bytes: float4 ((ch * 4 + q) * 4 + v) * 32 + lane.  sum_part2: this
      // lane's 16 values of chunks ch and ch + 2, both halves added (all
      // four loads issued before the first add).
      auto sum_part2 = [&](uint32_t (&r0)[16], uint32_t (&r1)[16], int ch) {
        const float4* const a = reinterpret_cast<const float4*>(p.part) + (ch * 4 + q) * 128 + lane;
        const float4* const b = a + 8 * 128;  // chunk ch + 2
        uint32_t o0[16], o1[16];
        ld_part16(a + part_of(tc.kh), r0);
        ld_part16(b + part_of(tc.kh), r1);
        ld_part16(a + part_of(tc.kh ^ 1), o0);
        ld_part16(b + part_of(tc.kh ^ 1), o1);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          r0[j] = __float_as_uint(__uint_as_float(r0[j]) + __uint_as_float(o0[j]));
          r1[j] = __float_as_uint(__uint_as_float(r1[j]) + __uint_as_float(o1[j]));
        }
      };
      // src 1, after its own partial sum is out: the claimant's.  One lane
      // waits for the flag (the claimant is past its MMAs and depends on no
      // other CTA, so the bounded wait ends); every epilogue thread takes the
      // verdict (false: an abandoned pipeline, whose error word is set).
      auto await_part = [&]() -> bool {
        uint32_t ok = 1;
        if (warp == kEpiWarp0 && lane == 0)
          ok = wait_flag_gpu(p.ks_cnt + 4 * tc.ks + 2 * crank + 1, p, abort_flag, 19u) ? 1u : 0u;
        return epi_barrier_and(ok) != 0u;
      };
      // src 1 and 2: the whole accumulator out to this half's buffer, in the
      // 16-bit path's round order (a slot's shared columns first) and with
      // its releases
      auto drain_partial = [&]() {
        constexpr int kNch = kCols / 16;
        auto group_of = [&](int k) { return slot == 0 ? 3 - k : k; };
        auto chunk_of = [&](int c0_, int i) { return 4 * group_of(c0_ / 2 + i / 2) + 2 * (i & 1) + h; };
        uint32_t rb[kRnd][16];
#pragma unroll
        for (int c0 = 0; c0 < kNch; c0 += kRnd) {
#pragma unroll
          for (int i = 0; i < kRnd; ++i) tc_ld_32x32b_x16(tbase + 16 * chunk_of(c0, i), rb[i]);
          tc_wait_ld();
          if (c0 == 0) release_shared();
          if (c0 + kRnd >= kNch) release();
#pragma unroll
          for (int i = 0; i < kRnd; ++i) {
            float4* const d = reinterpret_cast<float4*>(p.part) + part_of(tc.kh) + (chunk_of(c0, i) * 4 + q) * 128 + lane;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              d[32 * v] = make_float4(__uint_as_float(rb[i][4 * v]), __uint_as_float(rb[i][4 * v + 1]),
                                      __uint_as_float(rb[i][4 * v + 2]), __uint_as_float(rb[i][4 * v + 3]));
          }
        }
      };
      // kOvl units (FP8 operands, so 16-bit or fp32 C): warp h drains the
      // unit's 16-column chunks h, h + 2, h + 4, ...; a whole unit in slot 0
      // takes its chunks in the columns shared with slot 1 (its last 80:
      // chunks 11..15) first, so that the first round of loads frees them
      // (in slot 1 they are the first chunks already).  A half-width unit is
      // always a CTA's last: no unit waits on its shared columns.
      //
      // 16-bit n-major C leaves in whole 128-byte row pieces: the two warps
      // of a lane quarter each hold two of a 64-column group's four chunks,
      // put them in the quarter's 4 KB staging buffer and, after a barrier
      // of the pair, each stores 16 of its 32 rows.  A store request then
      // covers a whole 128-byte line, not one 32-byte sector of 16 lines,
      // and those scattered sector writes measurably slowed the next unit's
      // operand loads.
      auto drain_overlapped = [&](auto cw_tag, int n_end) {
        constexpr int CW = decltype(cw_tag)::value;
        constexpr int kNch = CW / 16;  // chunks of this warp: 8, or 4 in a half-width unit
        static_assert(kNch == 8 || kNch == 4, "whole or half 256-wide unit");
        const int rot = (CW == kCols && slot == 0) ? (h ? 5 : 6) : 0;
        // the unit column of drain slot s
        auto col_of = [&](int s_) { return 16 * (2 * ((rot + s_) & (kNch - 1)) + h); };
        const int row0 = tc.mt * kTileM + q * 32;
        if (p.c_dtype != BSG_F32) {
          // 16-bit C: each round of chunks rounded, packed and stored as it
          // leaves tensor memory.  Only the first round's release (the shared
          // columns) is on the next unit's path; the full release is needed
          // one unit later, so the rounds need not all stay in registers.
          // A round is two 64-column groups; slot 0 takes a whole unit's
          // groups from the last (its shared chunks 11..15 lie in groups 2
          // and 3), slot 1 and half-width units from the first.
          auto group_of = [&](int k) { return (CW == kCols && slot == 0) ? 3 - k : k; };
          // chunk held in round slot i of the round starting at slot c0
          auto chunk_of = [&](int c0_, int i) { return 4 * group_of(c0_ / 2 + i / 2) + 2 * (i & 1) + h; };
          uint32_t rb[kRnd][16];
          const bool bf = p.c_dtype == BSG_BF16;
          uint16_t* const cbase = static_cast<uint16_t*>(p.c) + batch_off;
          uint8_t* const qstg = smem + p.smem_epi + q * (2 * kEpiStageBytes);
          // chunk ch of the unit (piece pair e of its 64-column group):
          // rounded, packed, counted toward Amax, and staged (n-major) or
          // stored (m-major)
          auto emit16 = [&](const uint32_t* r, int ch, int e) {
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float f0 = __uint_as_float(r[2 * j]), f1 = __uint_as_float(r[2 * j + 1]);
              if (bf) {
                const __nv_bfloat162 v = __floats2bfloat162_rn(f0, f1);
                w[j] = *reinterpret_cast<const uint32_t*>(&v);
              } else {
                const __half2 v = __floats2half2_rn(f0, f1);
                w[j] = *reinterpret_cast<const uint32_t*>(&v);
              }
            }
            const int col = ucol0 + 16 * ch;
            // only stored elements count toward Amax
            const int nv = row_ok ? n_end - col : 0;
            if (nv >= 16) {
#pragma unroll
              for (int j = 0; j < 8; ++j) vmax = __vmaxu2(vmax, w[j] & 0x7FFF7FFFu);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                uint32_t m = w[j] & 0x7FFF7FFFu;
                if (2 * j >= nv) m &= 0xFFFF0000u;
                if (2 * j + 1 >= nv) m &= 0x0000FFFFu;
                vmax = __vmaxu2(vmax, m);
              }
            }
            if (p.c_major == 0) {
              // this row's 32 bytes of the chunk: 16-byte pieces
              // 2(2e + h) and 2(2e + h) + 1 of the 128-byte staged row,
              // XOR-swizzled by row % 8 (conflict-free both ways)
              const int pc0 = 2 * (2 * e + h);
              uint8_t* const srow = qstg + lane * 128;
              *reinterpret_cast<uint4*>(srow + ((pc0 ^ (lane & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(srow + (((pc0 + 1) ^ (lane & 7)) * 16)) =
                  make_uint4(w[4], w[5], w[6], w[7]);
            } else {
              // m-major: column by column, the 32 lanes write 32 consecutive rows
              uint16_t* dst = cbase + static_cast<size_t>(col) * p.M + row;
              const int ncols = row_ok ? min(16, n_end - col) : 0;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (j < ncols)
                  *dst = static_cast<uint16_t>((j & 1) ? (w[j / 2] >> 16) : (w[j / 2] & 0xFFFFu));
                dst += p.M;
              }
            }
          };
          // n-major: the staged 64-column group g out, 32 rows x 128 bytes;
          // this warp stores rows 16h .. 16h + 15, four rows (eight lanes
          // each) per store
          auto store_group = [&](int g) {
            if (p.c_major != 0) return;
            named_bar_sync(2 + q, 64);
            const int gcol = ucol0 + 64 * g;
            const int bytes_valid = (n_end - gcol) * 2;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int rr = 16 * h + 4 * j + (lane >> 3), pc = lane & 7;
              const uint4 x = *reinterpret_cast<const uint4*>(qstg + rr * 128 + ((pc ^ (rr & 7)) * 16));
              if (row0 + rr < p.M && pc * 16 < bytes_valid)
                *reinterpret_cast<uint4*>(reinterpret_cast<char*>(
                    cbase + static_cast<size_t>(row0 + rr) * p.N + gcol) + pc * 16) = x;
            }
            named_bar_sync(2 + q, 64);  // the buffer is free for the next group
          };
          if (!kKs || src == 0) {
#pragma unroll
            for (int c0 = 0; c0 < kNch; c0 += kRnd) {
#pragma unroll
              for (int i = 0; i < kRnd; ++i) tc_ld_32x32b_x16(tbase + 16 * chunk_of(c0, i), rb[i]);
              tc_wait_ld();
              if (c0 == 0) release_shared();
              if (c0 + kRnd >= kNch) release();
#pragma unroll
              for (int k = 0; k < kRnd / 2; ++k) {
#pragma unroll
                for (int e = 0; e < 2; ++e) emit16(rb[2 * k + e], chunk_of(c0, 2 * k + e), e);
                store_group(group_of(c0 / 2 + k));
              }
            }
          } else {
            // a K half: C from the two partial sums, a 64-column group at a
            // time (its two chunks' loads in flight together)
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
              uint32_t r0[16], r1[16];
              sum_part2(r0, r1, 4 * g + h);
              emit16(r0, 4 * g + h, 0);
              emit16(r1, 4 * g + 2 + h, 1);
              store_group(g);
            }
          }
        } else {
          // fp32 C: the first half of the slots in registers; each goes out
          // (n-major through the staging buffer, m-major column by column)
          // and the second half's chunk is loaded into its registers
          float* const cbase = static_cast<float*>(p.c) + batch_off;
          constexpr int kP1 = kNch / 2;
          auto chunk_out = [&](int col, const uint32_t* rr) {
            const int nv = n_end - col;  // the chunk's stored columns
            if (row_ok && nv >= 16) {
#pragma unroll
              for (int j = 0; j < 16; ++j) vmax = max(vmax, rr[j] & 0x7FFFFFFFu);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (row_ok && j < nv) vmax = max(vmax, rr[j] & 0x7FFFFFFFu);
            }
            if (p.c_major == 0) {
              char* const g = reinterpret_cast<char*>(cbase + static_cast<size_t>(row0) * p.N + col);
              store_rows_coalesced<16>(stg, rr, lane, g, static_cast<size_t>(p.N) * 4, p.M - row0,
                                       nv * 4);
            } else {
              float* dst = cbase + static_cast<size_t>(col) * p.M + row;
              const int ncols = row_ok ? min(16, nv) : 0;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (j < ncols) *dst = __uint_as_float(rr[j]);
                dst += p.M;
              }
            }
          };
          uint32_t r[kP1 * 16];
          if (!kKs || src == 0) {
#pragma unroll
            for (int i = 0; i < kP1; ++i) tc_ld_32x32b_x16(tbase + col_of(i), r + 16 * i);
            tc_wait_ld();
            // a whole unit's shared chunks are among its first kP1 slots
            if (CW == kCols) release_shared();
#pragma unroll
            for (int i = 0; i < kP1; ++i) {
              chunk_out(ucol0 + col_of(i), r + 16 * i);
              tc_ld_32x32b_x16(tbase + col_of(kP1 + i), r + 16 * i);
            }
            tc_wait_ld();
            if (CW != kCols) release_shared();
            release();
#pragma unroll
            for (int i = 0; i < kP1; ++i) chunk_out(ucol0 + col_of(kP1 + i), r + 16 * i);
          } else {
            // a K half: C from the two partial sums, two chunks at a time
            // (their loads in flight together)
#pragma unroll 1
            for (int ch = h; ch < 2 * kNch; ch += 4) {
              uint32_t r0[16], r1[16];
              sum_part2(r0, r1, ch);
              chunk_out(ucol0 + 16 * ch, r0);
              chunk_out(ucol0 + 16 * (ch + 2), r1);
            }
          }
        }
      };
      // the unit's stores: CW accumulator columns per warp, a compile-time
      // width (a runtime one spilled registers in these unrolled loops)
      auto unit = [&](auto cw_tag) {
        constexpr int CW = decltype(cw_tag)::value;  // columns of this warp in this unit
        const int n_end = min(p.N, ucol0 + 2 * CW);   // one past the unit's last stored column
        if constexpr (kOvl) {
          drain_overlapped(std::integral_constant<int, CW>{}, n_end);
        } else {
          constexpr int kChU = CW / 16;                 // its 16-column chunks
          const uint32_t taddr = tbase + h * CW;
          const int n0 = ucol0 + h * CW;
          // columns of this warp's part stored in this lane's row (may be <= 0)
          const int lim = row_ok ? n_end - n0 : 0;
          // one round of tensor-memory loads
          uint32_t rb[kRnd][16];
          if constexpr (LOWC) {
            // FP8 or packed E2M1 C (FP4 operands only): each round of kRnd
            // 16-column chunks is converted as it leaves tensor memory and
            // stored at once (holding every code of the warp's columns until
            // the end spilled registers); Amax is the rounded value of the
            // largest stored magnitude (the rounding is monotone in |x|)
            const bool fp4 = p.c_dtype == BSG_E2M1, e5 = p.c_dtype == BSG_E5M2;
            constexpr int kRc = kRnd * 16;  // columns per round
            uint8_t* const cbase = static_cast<uint8_t*>(p.c) + (fp4 ? batch_off / 2 : batch_off);
            const int row0 = tc.mt * kTileM + q * 32;
            const int ncols = row_ok ? min(CW, n_end - n0) : 0;  // m-major: stored columns
  #pragma unroll
            for (int c0 = 0; c0 < kChU; c0 += kRnd) {
  #pragma unroll
              for (int i = 0; i < kRnd; ++i)
                if (c0 + i < kChU) tc_ld_32x32b_x16(taddr + (c0 + i) * 16, rb[i]);
              tc_wait_ld();
              // the last round's loads have landed: free the accumulator before
              // converting them (the MMAs of the next unit wait for this)
              if (c0 + kRnd >= kChU) release();
              // the round's codes: four FP8 per word, or eight E2M1 (the first
              // kRc / 8 words)
              uint32_t pr[kRc / 4];
  #pragma unroll
              for (int i = 0; i < kRnd; ++i) {
                const int cc = (c0 + i) * 16;
                const uint32_t* r = rb[i];
                if (lim >= cc + 16) {
  #pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    uint32_t a = r[j] & 0x7FFFFFFFu;
                    if (fp4 && a > 0x7F800000u) a = 0u;  // stored as +0
                    vmax = max(vmax, a);
                  }
                } else {
  #pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    uint32_t a = r[j] & 0x7FFFFFFFu;
                    if (fp4 && a > 0x7F800000u) a = 0u;
                    if (cc + j >= lim) a = 0u;
                    vmax = max(vmax, a);
                  }
                }
                if (fp4) {
                  uint32_t w0 = 0u, w1 = 0u;
  #pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    const uint32_t b = cvt2_e2m1(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                    if (j < 4) w0 |= b << (8 * j);
                    else w1 |= b << (8 * (j - 4));
                  }
                  pr[2 * i] = w0;
                  pr[2 * i + 1] = w1;
                } else {
  #pragma unroll
                  for (int j = 0; j < 8; j += 2) {
                    const float a0 = __uint_as_float(r[2 * j]), a1 = __uint_as_float(r[2 * j + 1]);
                    const float b0 = __uint_as_float(r[2 * j + 2]), b1 = __uint_as_float(r[2 * j + 3]);
                    const uint32_t lo = e5 ? cvt2_e5m2(a0, a1) : cvt2_e4m3(a0, a1);
                    const uint32_t hi = e5 ? cvt2_e5m2(b0, b1) : cvt2_e4m3(b0, b1);
                    pr[4 * i + j / 2] = lo | (hi << 16);
                  }
                }
              }
              const int cr = c0 * 16;  // the round's first column in this warp's part
              if (p.c_major == 0) {
                if (fp4) {
                  // kRc / 2 bytes per row: one staged chunk of 8 words
                  char* const g = reinterpret_cast<char*>(
                      cbase + static_cast<size_t>(row0) * (p.N / 2) + (n0 + cr) / 2);
                  store_rows_coalesced<kRc / 8>(stg, pr, lane, g, static_cast<size_t>(p.N / 2),
                                                p.M - row0, (n_end - n0 - cr) / 2);
                } else {
                  char* const g = reinterpret_cast<char*>(cbase + static_cast<size_t>(row0) * p.N + n0 + cr);
                  store_rows_coalesced<kRc / 4>(stg, pr, lane, g, static_cast<size_t>(p.N), p.M - row0,
                                                n_end - n0 - cr);
                }
              } else {
                // m-major FP8: column by column, the 32 lanes write 32 consecutive rows
                uint8_t* dst = cbase + static_cast<size_t>(n0 + cr) * p.M + row;
  #pragma unroll
                for (int j = 0; j < kRc; ++j) {
                  if (cr + j < ncols) *dst = static_cast<uint8_t>(pr[j / 4] >> (8 * (j % 4)));
                  dst += p.M;
                }
              }
            }
          } else if (p.c_dtype != BSG_F32) {
            uint32_t pk[CW / 2];
            // pk: two rounded 16-bit values per register
            const bool bf = p.c_dtype == BSG_BF16;
            // rounds of kRnd 16-column loads: all of a round in flight at once,
            // one wait, then its conversions (fewer waits than one load ahead)
  #pragma unroll
            for (int c0 = 0; c0 < kChU; c0 += kRnd) {
  #pragma unroll
              for (int i = 0; i < kRnd; ++i)
                if (c0 + i < kChU) tc_ld_32x32b_x16(taddr + (c0 + i) * 16, rb[i]);
              tc_wait_ld();
              // the last round's loads have landed: free the accumulator before
              // converting them (the MMAs of the next unit wait for this)
              if (c0 + kRnd >= kChU) release();
  #pragma unroll
              for (int i = 0; i < kRnd; ++i) {
                if (c0 + i >= kChU) continue;
                const int cc = (c0 + i) * 16;
                const uint32_t* r = rb[i];
  #pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float f0 = __uint_as_float(r[2 * j]), f1 = __uint_as_float(r[2 * j + 1]);
                  // two round-to-nearest-even conversions in one: low half column
                  // cc + 2j, high half column cc + 2j + 1
                  uint32_t h;
                  if (bf) {
                    const __nv_bfloat162 v = __floats2bfloat162_rn(f0, f1);
                    h = *reinterpret_cast<const uint32_t*>(&v);
                  } else {
                    const __half2 v = __floats2half2_rn(f0, f1);
                    h = *reinterpret_cast<const uint32_t*>(&v);
                  }
                  pk[cc / 2 + j] = h;
                }
                // only stored elements count toward Amax: a whole chunk without
                // per-element tests (which made the drain four times slower),
                // the ragged edge with them
                if (lim >= cc + 16) {
  #pragma unroll
                  for (int j = 0; j < 8; ++j) vmax = __vmaxu2(vmax, pk[cc / 2 + j] & 0x7FFF7FFFu);
                } else {
  #pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    uint32_t m = pk[cc / 2 + j] & 0x7FFF7FFFu;
                    if (cc + 2 * j >= lim) m &= 0xFFFF0000u;
                    if (cc + 2 * j + 1 >= lim) m &= 0x0000FFFFu;
                    vmax = __vmaxu2(vmax, m);
                  }
                }
              }
            }
            uint16_t* const cbase = static_cast<uint16_t*>(p.c) + batch_off;
            if (p.c_major == 0) {
              // 32-column chunks (64 bytes per row) through the staging buffer;
              // a 112-column half ends with a 16-column chunk
              const int row0 = tc.mt * kTileM + q * 32;
              char* const g0 = reinterpret_cast<char*>(cbase + static_cast<size_t>(row0) * p.N + n0);
              const size_t pitch = static_cast<size_t>(p.N) * 2;
  #pragma unroll
              for (int cc = 0; cc + 32 <= CW; cc += 32)
                if (cc < CW)
                  store_rows_coalesced<16>(stg, pk + cc / 2, lane, g0 + cc * 2, pitch, p.M - row0,
                                           (n_end - n0 - cc) * 2);
              if (CW % 32 == 16)  // (never a half-width unit: those come from 256-wide tiles)
                store_rows_coalesced<8>(stg, pk + (CW - 16) / 2, lane, g0 + (CW - 16) * 2, pitch,
                                        p.M - row0, (n_end - n0 - (CW - 16)) * 2);
            } else {
              // m-major: column by column, the 32 lanes write 32 consecutive rows
              uint16_t* dst = cbase + static_cast<size_t>(n0) * p.M + row;
              const int ncols = row_ok ? min(CW, n_end - n0) : 0;
  #pragma unroll
              for (int j = 0; j < CW; ++j) {
                if (j < ncols)
                  *dst = static_cast<uint16_t>((j & 1) ? (pk[j / 2] >> 16) : (pk[j / 2] & 0xFFFFu));
                dst += p.M;
              }
            }
          } else {
            float* const cbase = static_cast<float*>(p.c) + batch_off;
            constexpr int kCh = CW / 16;         // 16-column chunks of this warp
            constexpr int kP1 = (kCh + 1) / 2;   // chunks held in registers at once
            constexpr int kP2 = kCh - kP1;       // the rest, loaded as the first go out
            // chunk ci (its 16 values in rr): Amax of the stored elements, then
            // the stores -- n-major through the staging buffer (64 bytes per
            // row), m-major column by column (32 consecutive rows per store)
            auto chunk_out = [&](int ci, const uint32_t* rr) {
              const int nb = n0 + 16 * ci;
              if (row_ok && nb + 16 <= n_end) {
  #pragma unroll
                for (int j = 0; j < 16; ++j) vmax = max(vmax, rr[j] & 0x7FFFFFFFu);
              } else {
  #pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (row_ok && nb + j < n_end) vmax = max(vmax, rr[j] & 0x7FFFFFFFu);
              }
              if (p.c_major == 0) {
                const int row0 = tc.mt * kTileM + q * 32;
                char* const g = reinterpret_cast<char*>(cbase + static_cast<size_t>(row0) * p.N + nb);
                store_rows_coalesced<16>(stg, rr, lane, g, static_cast<size_t>(p.N) * 4, p.M - row0,
                                         (n_end - nb) * 4);
              } else {
                float* dst = cbase + static_cast<size_t>(nb) * p.M + row;
                const int ncols = row_ok ? min(16, n_end - nb) : 0;
  #pragma unroll
                for (int j = 0; j < 16; ++j) {
                  if (j < ncols) *dst = __uint_as_float(rr[j]);
                  dst += p.M;
                }
              }
            };
            uint32_t r[kP1 * 16];
  #pragma unroll
            for (int i = 0; i < kP1; ++i) tc_ld_32x32b_x16(taddr + i * 16, r + 16 * i);
            tc_wait_ld();
            if (kP2 == 0) release();
            // each first chunk out, then the second half's chunk loaded into its
            // registers: the loads overlap the stores, and the accumulator is
            // freed as soon as the last of them lands
  #pragma unroll
            for (int i = 0; i < kP1; ++i) {
              chunk_out(i, r + 16 * i);
              if (i < kP2) tc_ld_32x32b_x16(taddr + (kP1 + i) * 16, r + 16 * i);
            }
            if (kP2 > 0) {
              tc_wait_ld();
              release();
  #pragma unroll
              for (int i = 0; i < kP2; ++i) chunk_out(kP1 + i, r + 16 * i);
            }
          }
        }
      };
      if constexpr (kKs) {
        if (tc.ks >= 0) {
          // both halves' partial sums go out; the claimant publishes its
          // own, the other half waits for it and stores C
          src = epi_barrier_and(ks_first) ? 2 : 1;
          drain_partial();
          if (src == 2) {
            // every thread's stores ordered before the flag
            __threadfence();
            epi_barrier_and(1u);
            if (warp == kEpiWarp0 && lane == 0) st_release_gpu(p.ks_cnt + 4 * tc.ks + 2 * crank + 1, 1u);
            continue;
          }
          if (!await_part()) continue;
        }
      }
      if constexpr (kHalves) {
        if (hu) unit(std::integral_constant<int, kCols / 2>{});
        else unit(std::integral_constant<int, kCols>{});
      } else {
        unit(std::integral_constant<int, kCols>{});
      }
    }
    if constexpr (LOWC) {
      // the stored magnitude of the largest |C|: round it like the stores did
      const float mx = __uint_as_float(vmax);
      const uint32_t code = p.c_dtype == BSG_E2M1 ? cvt2_e2m1(mx, 0.0f) & 0xFu
                            : p.c_dtype == BSG_E5M2 ? cvt2_e5m2(mx, 0.0f) & 0xFFu
                                                    : cvt2_e4m3(mx, 0.0f) & 0xFFu;
      vmax = abs_bits_f32(decode_mag(code, p.c_dtype));
    } else if (p.c_dtype != BSG_F32) {
      const uint32_t hmax = max(vmax & 0xFFFFu, vmax >> 16);
      vmax = p.c_dtype == BSG_BF16
                 ? hmax << 16
                 : abs_bits_f32(__half2float(__ushort_as_half(static_cast<unsigned short>(hmax))));
    }
    vmax = __reduce_max_sync(0xFFFFFFFFu, vmax);
    if (lane == 0) atomicMax(cta_amax, vmax);
  }

  tc_fence_before();
  if (CM > 1 && !cl_arrived) {
    __syncwarp();
    cluster_arrive();
  }
  __syncthreads();
  if (CM > 1) cluster_wait();  // the peer arrives into this CTA no more
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols)
                   : "memory");
  }
  if (threadIdx.x == 0) {
    // global Amax: max over CTAs, written by the last CTA to arrive, which
    // also re-zeroes the two workspace slots and the K halves' words for the
    // next run (every CTA is past its epilogue by then, an abandoned launch
    // too)
    atomicMax(p.ws + 0, *cta_amax);
    __threadfence();
    const uint32_t arrived = atomicAdd(p.ws + 1, 1u);
    if (arrived == gridDim.x - 1) {
      __threadfence();
      const uint32_t bits = atomicExch(p.ws + 0, 0u);
      *p.amax = __uint_as_float(bits);
      if constexpr (kKs)
        for (int i = 0; i < 4 * p.ks_tiles; ++i) p.ks_cnt[i] = 0u;
      atomicExch(p.ws + 1, 0u);
    }
  }
}
#undef BSG_WAIT
#undef BSG_WAIT_SLEEP

// Kernel variants: MMA kind x (TILE_N, accumulator buffers) x cluster along M
// (cm 1: a CTA alone; 2: a cta_group::2 pair)
struct Variant {
  int kind, tile_n, num_acc, cm, pair, kslices, lowc, kspl;
  const void* fn;
};

template <int KIND, int TN, int NACC, int CM, int PAIR, int LOWC = 0, int KSL = 1, int KSPL = 0>
Variant make_variant() {
  return Variant{KIND, TN, NACC, CM, PAIR, KSL, LOWC, KSPL,
                 reinterpret_cast<const void*>(
                     &bsg_gemm_amax_kernel<KIND, TN, NACC, CM, PAIR, KSL, LOWC, KSPL>)};
}

template <int KIND, int LOWC>
void add_kind(Variant* out, int& n) {
  out[n++] = make_variant<KIND, 128, 2, 1, 0, LOWC>();
  out[n++] = make_variant<KIND, 256, 1, 1, 0, LOWC>();
  out[n++] = make_variant<KIND, 256, 1, 2, 1, LOWC>();
}

const Variant* find_variant(int kind, int tile_n, int num_acc, int cm, int kslices, int lowc,
                            int kspl = 0) {
  static Variant table[24];
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    add_kind<kKindF8F6F4, 0>(table, n);
    table[n++] = make_variant<kKindF8F6F4, 224, 2, 2, 1>();  // 256 x 224 pairs, two accumulators
    table[n++] = make_variant<kKindF8F6F4, 256, 1, 2, 1, 0, 1, 1>();  // pairs with K halves
    add_kind<kKindF4x4X, 0>(table, n);
    add_kind<kKindF4x2X, 0>(table, n);
    add_kind<kKindF4x4X, 1>(table, n);  // FP4 operands with E4M3 / E5M2 / E2M1 C
    add_kind<kKindF4x2X, 1>(table, n);
  });
  for (int i = 0; i < n; ++i) {
    const Variant& v = table[i];
    if (v.kind == kind && v.tile_n == tile_n && v.num_acc == num_acc && v.cm == cm &&
        v.kslices == kslices && v.lowc == lowc && v.kspl == kspl)
      return &v;
  }
  return nullptr;
}

// ------------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

constexpr size_t kWorkspaceBytes = 256;
// Past those words, for a plan with K halves: two words per split tile and
// CTA rank (halves claimed, partial sum out; rounded up to 256 bytes), then
// per split tile, K half and CTA rank a 128 x 256 fp32 partial sum.
constexpr size_t kPartBytes = static_cast<size_t>(128) * 256 * 4;
inline size_t ks_cnt_bytes(int tiles) { return (static_cast<size_t>(16) * tiles + 255) / 256 * 256; }
inline size_t ws_need(int ks_tiles) {
  return ks_tiles ? kWorkspaceBytes + ks_cnt_bytes(ks_tiles) + static_cast<size_t>(ks_tiles) * 4 * kPartBytes
                  : kWorkspaceBytes;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
// bytes of C's contiguous extent of `n` elements
inline int64_t c_extent_bytes(int64_t n, int d) {
  switch (d) {
    case BSG_F32: return n * 4;
    case BSG_F16:
    case BSG_BF16: return n * 2;
    case BSG_E2M1: return n / 2;
    default: return n;  // FP8
  }
}

}  // namespace

struct bsg_plan {
  bsg_problem prob;
  int device;
  int sm_count;
  Params base;           // everything but the pointers
  const void* kernel;    // the chosen kernel variant
  const void* kernel_ks; // its instantiation with K halves (plans with k_split_tiles)
  int kind;
  int num_acc;
  int cluster_m;         // CTAs per cluster along M: 1, or 2 for a cta_group::2 pair
  int kslices;           // 128-byte K slices per pipeline stage
  int pair;              // 1: the cluster is a cta_group::2 pair (256-row MMAs)
  int half_tiles;        // tiles of the last wave run as two half-width units
  int ks_tiles;          // tiles past the whole waves run as two K halves (a full workspace)
  int max_clusters;      // clusters resident at once (persistent launches of pairs)
  size_t ws_bytes;       // workspace of the plan's fastest form (with the K halves' buffers)
  int grid;
  int smem_bytes;
  // tensor maps for the last A/B pointers seen
  std::mutex mu;
  const void* map_a_ptr = nullptr;
  const void* map_b_ptr = nullptr;
  const void* map_sfa_ptr = nullptr;
  const void* map_sfb_ptr = nullptr;
  const void* map_bh_ptr = nullptr;
  CUtensorMap map_a;
  CUtensorMap map_b;
  CUtensorMap map_bh;    // B with the half-width units' 64-row box
  CUtensorMap map_sfa;
  CUtensorMap map_sfb;
};

// The schedule of one launch, by the workspace it is given: K halves when it
// holds their buffers, else the half-width split of the last wave, else
// whole tiles alone.
static Params launch_params(const bsg_plan* plan, size_t ws_bytes) {
  Params k = plan->base;
  const int tiles = k.num_units;
  if (plan->ks_tiles && ws_bytes >= plan->ws_bytes) {
    k.ks_tiles = plan->ks_tiles;
    k.ks_k0 = k.k_stages / 2;
    k.ks_first = tiles - plan->ks_tiles;
    k.num_units = tiles + plan->ks_tiles;
    k.full_units = k.num_units;
  } else if (plan->half_tiles) {
    k.full_units = tiles - plan->half_tiles;
    k.num_units = k.full_units + 2 * plan->half_tiles;
  }
  return k;
}

// CTAs of that launch: persistent clusters, at most as many as are resident
static int launch_grid(const bsg_plan* plan, const Params& k) {
  if (plan->cluster_m > 1) {
    const int clusters = k.num_units < plan->max_clusters ? k.num_units : plan->max_clusters;
    return plan->cluster_m * clusters;
  }
  return k.num_units < plan->sm_count ? k.num_units : plan->sm_count;
}

extern "C" {

const char* bsg_status_string(bsg_status s) {
  switch (s) {
    case BSG_OK: return "ok";
    case BSG_ERR_INVALID_ARG: return "invalid argument";
    case BSG_ERR_UNSUPPORTED: return "unsupported combination";
    case BSG_ERR_ALIGNMENT: return "misaligned pointer or row (16 bytes required)";
    case BSG_ERR_ARCH: return "device is not sm_103 (compute capability 10.3)";
    case BSG_ERR_WORKSPACE: return "workspace missing or too small";
    case BSG_ERR_CUDA: return "CUDA call failed";
    case BSG_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait timed out";
  }
  return "unknown status";
}

bsg_status bsg_problem_check(const bsg_problem* p) {
  if (!p) return BSG_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (p->M < 1 || p->N < 1 || p->K < 1 || p->L < 1) return BSG_ERR_INVALID_ARG;
  if (p->M > lim || p->N > lim || p->K > lim || p->L > lim) return BSG_ERR_INVALID_ARG;
  const int ops[2] = {p->a_dtype, p->b_dtype};
  for (int d : ops)
    if (d != BSG_E4M3 && d != BSG_E5M2 && d != BSG_E2M1) return BSG_ERR_INVALID_ARG;
  if (p->sf_dtype != BSG_UE8M0 && p->sf_dtype != BSG_E4M3) return BSG_ERR_INVALID_ARG;
  const bool c_low = p->c_dtype == BSG_E4M3 || p->c_dtype == BSG_E5M2 || p->c_dtype == BSG_E2M1;
  if (!c_low && p->c_dtype != BSG_F32 && p->c_dtype != BSG_F16 && p->c_dtype != BSG_BF16)
    return BSG_ERR_INVALID_ARG;
  if (p->sf_vec_size != 16 && p->sf_vec_size != 32) return BSG_ERR_INVALID_ARG;
  const bool a4 = p->a_dtype == BSG_E2M1, b4 = p->b_dtype == BSG_E2M1;
  if (a4 != b4) return BSG_ERR_UNSUPPORTED;                  // FP4 x FP8
  // low-precision C ("Support surface", "Dtypes"): FP8 C with FP8 operands
  // is disabled, E2M1 C needs FP4 operands and an n-major C
  if (c_low && !a4) return BSG_ERR_UNSUPPORTED;
  if (!a4 && p->sf_vec_size == 16) return BSG_ERR_UNSUPPORTED;  // FP8 needs sfv 32
  // E4M3 scales ("Dtypes"): only the NVFP4 form, FP4 operands with sfv 16
  if (p->sf_dtype == BSG_E4M3 && (!a4 || p->sf_vec_size != 16)) return BSG_ERR_UNSUPPORTED;
  // operand majors ("Parameters": A k- or m-major, B k- or n-major; packed
  // FP4 k-major only)
  if (p->a_major != 'k' && p->a_major != 'm') return BSG_ERR_INVALID_ARG;
  if (p->b_major != 'k' && p->b_major != 'n') return BSG_ERR_INVALID_ARG;
  const bool a_mn = p->a_major == 'm', b_mn = p->b_major == 'n';
  if ((a_mn || b_mn) && a4) return BSG_ERR_UNSUPPORTED;
  if (p->c_major != 'n' && p->c_major != 'm') return BSG_ERR_INVALID_ARG;
  if (p->c_dtype == BSG_E2M1 && p->c_major != 'n') return BSG_ERR_UNSUPPORTED;
  if (p->tile_m != 0 && p->tile_m != 128) return BSG_ERR_INVALID_ARG;
  if (p->tile_n != 0 && p->tile_n != 128 && p->tile_n != 224 && p->tile_n != 256)
    return BSG_ERR_INVALID_ARG;
  const int cl[2] = {p->cluster_m, p->cluster_n};
  for (int c : cl)
    if (c != 0 && c != 1 && c != 2 && c != 4) return BSG_ERR_INVALID_ARG;
  // clusters: one CTA, or a cta_group::2 pair along M.  Larger clusters (the
  // page's cluster shapes that share a tile between CTAs by multicast) and
  // clusters along N are not built.
  if (p->cluster_m == 4 || p->cluster_n > 1) return BSG_ERR_UNSUPPORTED;
  // an n-major B tile is loaded whole by one CTA (single 128-wide tiles) or
  // in halves by a CTA pair; 256 columns in one CTA are k-major only
  if (b_mn && p->cluster_m == 1 && p->tile_n > 128) return BSG_ERR_UNSUPPORTED;
  const int64_t row_bytes = a4 ? p->K / 2 : p->K;
  if (a4 && (p->K % 2)) return BSG_ERR_ALIGNMENT;
  // the contiguous extent of each operand: K bytes, or M (N) bytes per K
  if ((!a_mn || !b_mn) && (row_bytes % 16)) return BSG_ERR_ALIGNMENT;
  if ((a_mn && p->M % 16) || (b_mn && p->N % 16)) return BSG_ERR_ALIGNMENT;
  const int64_t c_n = p->c_major == 'n' ? p->N : p->M;
  if (p->c_dtype == BSG_E2M1 && (c_n % 2)) return BSG_ERR_ALIGNMENT;
  if (c_extent_bytes(c_n, p->c_dtype) % 16) return BSG_ERR_ALIGNMENT;
  return BSG_OK;
}

bsg_status bsg_plan_create(const bsg_problem* prob, int device, bsg_plan** out) {
  if (!out) return BSG_ERR_INVALID_ARG;
  const bsg_status st = bsg_problem_check(prob);
  if (st != BSG_OK) return st;
  int major = 0, minor = 0, sms = 0, max_smem = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
          cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return BSG_ERR_ARCH;
  if (!get_encode_fn()) return BSG_ERR_CUDA;

  bsg_plan* plan = new (std::nothrow) bsg_plan();
  if (!plan) return BSG_ERR_INVALID_ARG;
  plan->prob = *prob;
  plan->device = device;
  plan->sm_count = sms;

  Params& k = plan->base;
  std::memset(&k, 0, sizeof(k));
  const bool fp4 = prob->a_dtype == BSG_E2M1;
  const int sfv = prob->sf_vec_size;
  k.M = static_cast<int>(prob->M);
  k.N = static_cast<int>(prob->N);
  k.K = static_cast<int>(prob->K);
  k.L = static_cast<int>(prob->L);
  int kind;
  if (!fp4) kind = kKindF8F6F4;          // one scale (block 32) per MMA: byte j of the column
  else if (sfv == 16) kind = kKindF4x4X;  // four block-16 scales per MMA: the whole column
  else kind = kKindF4x2X;                 // two block-32 scales per MMA: bytes 0-1 or 2-3
  const int chunks = kind == kKindF8F6F4 ? 1 : (kind == kKindF4x4X ? 4 : 2);
  k.tiles_m = static_cast<int>(cdiv(prob->M, kTileM));
  k.k_bytes = static_cast<int>(fp4 ? prob->K / 2 : prob->K);
  k.k_stages = static_cast<int>(cdiv(k.k_bytes, kStageKBytes));
  // Tile width.  256 (one accumulator) halves the issue work and the L2
  // traffic per flop against 128, and is the default above N = 128.  224
  // (FP8, CTA pairs only; a hint) keeps two accumulators in tensor memory so
  // that the epilogue overlaps the next tile; since the epilogue's drain of a
  // single accumulator became short, 256 measures faster on every workload
  // (MXFP8 4096^3: 2165 against 2035 TFLOP/s).
  const bool pair_ok = k.tiles_m >= 2 && (prob->cluster_m == 0 || prob->cluster_m == 2);
  const bool n224_ok = kind == kKindF8F6F4 && pair_ok;
  if (prob->tile_n == 128) {
    k.tile_n = 128;
  } else if (prob->tile_n == 256) {
    k.tile_n = 256;
  } else if (prob->tile_n == 224) {
    if (!n224_ok) { delete plan; return BSG_ERR_UNSUPPORTED; }
    k.tile_n = 224;
  } else {
    // small problems (128 x 128 tiles filling at most half of the SMs) run as
    // 128-wide single CTAs: the work is latency-bound and a single CTA needs
    // no cluster launch (E4M3 256^3: 10.8 against 14.3 us as a pair)
    const int64_t tiles128 = k.tiles_m * cdiv(prob->N, 128) * prob->L;
    const bool small = prob->cluster_m == 0 && tiles128 * 2 <= sms;
    k.tile_n = prob->N <= 128 || small ? 128 : 256;
  }
  int num_acc = k.tile_n == 256 ? 1 : 2;
  // 224- and 256-wide tiles run as cta_group::2 pairs by default (hint 1:
  // single CTAs; 224 is pairs only); the 128-wide variant runs alone
  int cm = 1;
  if (k.tile_n == 256) cm = prob->cluster_m == 0 ? 2 : prob->cluster_m;
  if (k.tile_n == 224) cm = 2;
  if (cm > k.tiles_m) cm = k.tiles_m >= 2 ? 2 : 1;
  const bool b_mn = prob->b_major == 'n';
  if (b_mn && cm == 1 && k.tile_n > 128) {
    // a single CTA holds at most one 128-column MN-major B tile
    if (prob->tile_n != 0) { delete plan; return BSG_ERR_UNSUPPORTED; }
    k.tile_n = 128;
    num_acc = 2;
  }
  // 128-byte K stages throughout: with the MMAs issued warp-wide the
  // per-stage cost is small, and more, smaller stages keep more operand
  // bytes in flight (256-byte stages measured 10 % slower at 4096^3)
  const int ksl = 1;
  const int stage_k_bytes = kStageKBytes * ksl;
  k.k_stages = static_cast<int>(cdiv(k.k_bytes, stage_k_bytes));
  const int lowc = prob->c_dtype == BSG_E4M3 || prob->c_dtype == BSG_E5M2 ||
                   prob->c_dtype == BSG_E2M1;
  const Variant* var = find_variant(kind, k.tile_n, num_acc, cm, ksl, lowc);
  if (!var) { delete plan; return BSG_ERR_UNSUPPORTED; }
  plan->kslices = ksl;
  plan->kernel = var->fn;
  plan->kind = kind;
  plan->num_acc = num_acc;
  plan->cluster_m = cm;
  plan->pair = var->pair;
  k.tiles_n = static_cast<int>(cdiv(prob->N, k.tile_n));
  k.num_tiles = k.tiles_m * k.tiles_n * k.L;
  k.tiles_mc = static_cast<int>(cdiv(k.tiles_m, cm));
  k.num_units = k.tiles_mc * k.tiles_n * k.L;
  k.full_units = k.num_units;
  k.t_m = static_cast<int>(cdiv(prob->M, 128));
  k.t_n = static_cast<int>(cdiv(prob->N, 128));
  k.t_k = static_cast<int>(cdiv(prob->K, 4 * sfv));
  uint32_t a_fmt, b_fmt;
  if (fp4) {
    a_fmt = b_fmt = 1;  // E2M1 in kind::mxf4nvf4
  } else {
    a_fmt = prob->a_dtype == BSG_E5M2 ? 1 : 0;  // kind::mxf8f6f4: E4M3 0, E5M2 1
    b_fmt = prob->b_dtype == BSG_E5M2 ? 1 : 0;
  }
  const int mma_m = plan->pair ? 2 * kTileM : kTileM;
  k.a_mn = prob->a_major == 'm' ? 1 : 0;
  k.b_mn = b_mn ? 1 : 0;
  // bits 15 / 16: A / B transposed, i.e. MN-major in shared memory
  k.idesc = (a_fmt << 7) | (b_fmt << 10) | (static_cast<uint32_t>(k.a_mn) << 15) |
            (static_cast<uint32_t>(k.b_mn) << 16) | (static_cast<uint32_t>(k.tile_n >> 3) << 17) |
            (prob->sf_dtype == BSG_UE8M0 ? 1u << 23 : 0u) /* scale type: 1 UE8M0, 0 UE4M3 */ |
            (static_cast<uint32_t>(mma_m >> 4) << 24);
  k.idesc_half = (k.idesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(k.tile_n >> 4) << 17);
  k.c_dtype = prob->c_dtype;
  k.c_major = prob->c_major == 'm' ? 1 : 0;

  const int G = (k.tile_n + 127) / 128;                       // scale groups the MMA reads
  const int sfb_atoms = k.tile_n % 128 == 0 ? G : G + 1;      // B scale atoms per chunk
  const int sfa_stage = chunks * ksl * kAtomBytes, sfb_stage = chunks * ksl * kAtomBytes * sfb_atoms;
  // B rows held per CTA: whole 128-row boxes (a 224-wide pair's half is loaded as 128 rows)
  const int b_rows = plan->pair ? (k.tile_n / 2 + 127) / 128 * 128 : k.tile_n;
  const int per_stage = kTileM * stage_k_bytes + b_rows * stage_k_bytes + sfa_stage + sfb_stage;
  const int reserve = 1024 /* alignment slack */ + 512 /* barriers and flags */ +
                      kEpiWarps * kEpiStageBytes /* epilogue staging */;
  int stages = (max_smem - reserve) / per_stage;
  if (stages > 8) stages = 8;
  const int sf_cols = 4 * chunks * ksl * (1 + G);
  // FP8 256-wide tiles with one accumulator use two overlapping accumulator
  // regions above the scale sets, which must fit in the 80 columns below
  const bool ovl = kind == kKindF8F6F4 && k.tile_n == 256 && num_acc == 1;
  const int tmem_need_acc = ovl ? 2 * k.tile_n - 80 : num_acc * k.tile_n;
  if (ovl)
    while (stages > 2 && stages * sf_cols > 80) --stages;
  while (stages > 2 && tmem_need_acc + stages * sf_cols > static_cast<int>(kTmemCols)) --stages;
  if (stages < 2 || tmem_need_acc + stages * sf_cols > static_cast<int>(kTmemCols) ||
      (ovl && stages * sf_cols > 80)) {
    delete plan;
    return BSG_ERR_UNSUPPORTED;
  }
  k.stages = stages;
  k.smem_a = 0;
  k.smem_b = k.smem_a + stages * kTileM * stage_k_bytes;
  k.smem_sfa = k.smem_b + stages * b_rows * stage_k_bytes;
  k.smem_sfb = k.smem_sfa + stages * sfa_stage;
  k.smem_epi = k.smem_sfb + stages * sfb_stage;
  k.smem_bar = k.smem_epi + kEpiWarps * kEpiStageBytes;
  // barriers: 5 per stage, 3 per accumulator slot (at most 2), the drain
  // and peer-record barriers, then 22 words of flags and the producers'
  // drain records; then the alignment slack
  plan->smem_bytes = static_cast<int>(k.smem_bar) + 40 * stages + 48 + 16 + 88 + 1024;
  k.wait_limit_ns = 1000000000ull;  // one second per wait
  if (const char* e = std::getenv("BSG_WAIT_LIMIT_NS")) {
    const unsigned long long v = std::strtoull(e, nullptr, 10);
    if (v > 0) k.wait_limit_ns = v;
  }
  plan->grid = k.num_units < sms ? k.num_units : sms;

  int prev = 0;
  cudaGetDevice(&prev);
  if (prev != device) cudaSetDevice(device);
  const cudaError_t e = cudaFuncSetAttribute(plan->kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             plan->smem_bytes);
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete plan;
    return BSG_ERR_CUDA;
  }
  if (cm > 1) {
    // persistent clusters: as many as can be resident at once
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cm;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(cm * (sms / cm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan->smem_bytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int max_clusters = 0;
    if (prev != device) cudaSetDevice(device);
    const cudaError_t oe = cudaOccupancyMaxActiveClusters(&max_clusters, plan->kernel, &cfg);
    if (prev != device) cudaSetDevice(prev);
    if (oe != cudaSuccess || max_clusters < 1) {
      cudaGetLastError();
      delete plan;
      return BSG_ERR_CUDA;
    }
    // The last wave: when the tiles left over after the full waves fill at
    // most half of the resident pairs, each runs as two half-width units
    // (256 x 128), so the final wave takes half a tile time.  256-wide pairs
    // with k-major B only (a 64-row box of an MN-major B is not a whole
    // 128-byte swizzle span).
    const int tail = k.num_units % max_clusters;
    if (plan->pair && k.tile_n == 256 && !b_mn && tail != 0 && 2 * tail <= max_clusters)
      plan->half_tiles = tail;
    // K halves, preferred where they apply (FP8 256-wide pairs, at least two
    // whole waves): every cluster then carries at most half a tile more than
    // the whole waves, at full width, where a half-width tile takes about as
    // long as a whole one.  The exchange of partial sums costs about as much
    // as 19 K stages, so they pay from 40 K stages on (the ragged L=2
    // workload, 56 stages: -2.6 %; 4096^3, 32 stages: +1.6 %, measured by
    // the benchmark's own timing).  BSG_KSPLIT_MIN_STAGES (read here) moves
    // that threshold, down to 2.  They need the workspace's partial-sum
    // buffers; a smaller workspace runs the half-width split (or none).
    int ks_min = 40;
    if (const char* e = std::getenv("BSG_KSPLIT_MIN_STAGES")) {
      const long v = std::strtol(e, nullptr, 10);
      if (v >= 2 && v <= (1L << 30)) ks_min = static_cast<int>(v);
    }
    if (plan->pair && kind == kKindF8F6F4 && k.tile_n == 256 && num_acc == 1 && tail != 0 &&
        2 * tail <= max_clusters && k.num_units / max_clusters >= 2 && k.k_stages >= ks_min) {
      const Variant* vk = find_variant(kind, k.tile_n, num_acc, cm, ksl, lowc, 1);
      if (vk) {
        if (prev != device) cudaSetDevice(device);
        const cudaError_t ek = cudaFuncSetAttribute(
            vk->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, plan->smem_bytes);
        if (prev != device) cudaSetDevice(prev);
        if (ek == cudaSuccess) {
          plan->kernel_ks = vk->fn;
          plan->ks_tiles = tail;
        } else {
          cudaGetLastError();
        }
      }
    }
    plan->max_clusters = max_clusters;
  }
  plan->ws_bytes = ws_need(plan->ks_tiles);
  {
    const Params f = launch_params(plan, plan->ws_bytes);
    plan->grid = launch_grid(plan, f);
  }
  if (std::getenv("BSG_LOG"))
    std::fprintf(stderr,
                 "[bsgemm] M=%lld N=%lld K=%lld L=%lld tile=128x%d stages=%d grid=%d smem=%d "
                 "kind=%d tiles=%d cluster_m=%d half_tiles=%d\n",
                 (long long)prob->M, (long long)prob->N, (long long)prob->K, (long long)prob->L,
                 k.tile_n, stages, plan->grid, plan->smem_bytes, kind, k.num_tiles, cm,
                 plan->half_tiles);
  *out = plan;
  return BSG_OK;
}

bsg_status bsg_plan_workspace_size(const bsg_plan* plan, size_t* bytes) {
  if (!plan || !bytes) return BSG_ERR_INVALID_ARG;
  *bytes = plan->ws_bytes;
  return BSG_OK;
}

bsg_status bsg_workspace_init(const bsg_plan* plan, void* ws, size_t ws_bytes, void* stream) {
  if (!plan || !ws) return BSG_ERR_INVALID_ARG;
  if (ws_bytes < kWorkspaceBytes) return BSG_ERR_WORKSPACE;
  // the words every run needs, and the K halves' counters when the
  // workspace is large enough for their form (the partial sums need no
  // initial value)
  const size_t zero = ws_bytes >= plan->ws_bytes && plan->ks_tiles
                          ? kWorkspaceBytes + ks_cnt_bytes(plan->ks_tiles)
                          : kWorkspaceBytes;
  if (cudaMemsetAsync(ws, 0, zero, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  return BSG_OK;
}

// An operand of `rows` rows and `k_bytes` bytes of K per row, batch
// outermost.  k-major: dims (K bytes, rows, L), box (one 128-byte K slice,
// box_rows rows).  MN-major (FP8; mn): dims (rows, K, L), box (box_rows
// MN bytes, one 128-row K slice) -- either way a 128-byte-swizzled box.
static bool encode_operand(CUtensorMap* map, const void* ptr, int64_t k_bytes, int64_t rows,
                           int64_t L, int box_rows, bool mn) {
  const int64_t inner = mn ? rows : k_bytes, outer = mn ? k_bytes : rows;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer),
                        static_cast<cuuint64_t>(L)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                           static_cast<cuuint64_t>(inner * outer)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(mn ? box_rows : kStageKBytes),
                       static_cast<cuuint32_t>(mn ? kStageKBytes : box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = get_encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr),
                                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Scale atoms as a 4-D tensor of 8-byte words: (64 words of one 512-byte
// atom, t_k atoms along K, t_mn atoms along M or N, L); the box is one
// stage's `k_atoms` K atoms of `mn_atoms` consecutive MN atoms.
static bool encode_scales(CUtensorMap* map, const void* ptr, int64_t t_k, int64_t t_mn, int64_t L,
                          int k_atoms, int mn_atoms) {
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(t_k), static_cast<cuuint64_t>(t_mn),
                        static_cast<cuuint64_t>(L)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kAtomBytes),
                           static_cast<cuuint64_t>(kAtomBytes * t_k),
                           static_cast<cuuint64_t>(kAtomBytes * t_k * t_mn)};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(k_atoms), static_cast<cuuint32_t>(mn_atoms), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = get_encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, const_cast<void*>(ptr),
                                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // extern "C"

namespace {

// The checks bsg_run makes on its tensor arguments before anything is
// enqueued: pointers present and aligned, and the plan's device current.
bsg_status check_run_args(const bsg_plan* plan, const void* A, const void* B, const void* SFA,
                          const void* SFB, const void* C, const float* amax) {
  if (!plan || !A || !B || !SFA || !SFB || !C || !amax) return BSG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(SFA) || !aligned16(SFB) || !aligned16(C) ||
      (reinterpret_cast<uintptr_t>(amax) & 3u))
    return BSG_ERR_ALIGNMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return BSG_ERR_CUDA; }
  if (dev != plan->device) return BSG_ERR_INVALID_ARG;
  return BSG_OK;
}

}  // namespace

extern "C" {

bsg_status bsg_run(const bsg_plan* cplan, const void* A, const void* B, const void* SFA,
                   const void* SFB, void* C, float* amax, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!cplan) return BSG_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kWorkspaceBytes || !aligned16(ws)) return BSG_ERR_WORKSPACE;
  const bsg_status arg_st = check_run_args(cplan, A, B, SFA, SFB, C, amax);
  if (arg_st != BSG_OK) return arg_st;
  bsg_plan* plan = const_cast<bsg_plan*>(cplan);
  const bsg_problem& pr = plan->prob;
  const int64_t row_bytes = plan->base.k_bytes;
  Params k = launch_params(plan, ws_bytes);
  if (k.ks_tiles) {
    char* const w = static_cast<char*>(ws);
    k.ks_cnt = reinterpret_cast<uint32_t*>(w + kWorkspaceBytes);
    k.part = reinterpret_cast<float*>(w + kWorkspaceBytes + ks_cnt_bytes(k.ks_tiles));
  }
  k.sfa = static_cast<const uint8_t*>(SFA);
  k.sfb = static_cast<const uint8_t*>(SFB);
  k.c = C;
  k.amax = amax;
  k.ws = static_cast<uint32_t*>(ws);
  CUtensorMap ma, mb, mbh, msfa, msfb;
  {
    std::lock_guard<std::mutex> lock(plan->mu);
    if (plan->map_a_ptr != A) {
      if (!encode_operand(&plan->map_a, A, row_bytes, pr.M, pr.L, kTileM, k.a_mn != 0)) {
        plan->map_a_ptr = nullptr;
        return BSG_ERR_CUDA;
      }
      plan->map_a_ptr = A;
    }
    if (plan->map_b_ptr != B) {
      const int b_box = plan->pair ? (k.tile_n / 2 + 127) / 128 * 128 : k.tile_n;
      if (!encode_operand(&plan->map_b, B, row_bytes, pr.N, pr.L, b_box, k.b_mn != 0)) {
        plan->map_b_ptr = nullptr;
        return BSG_ERR_CUDA;
      }
      plan->map_b_ptr = B;
    }
    if (k.full_units < k.num_units && plan->map_bh_ptr != B) {
      // each CTA of a pair loads 64 rows of a half-width unit's B
      if (!encode_operand(&plan->map_bh, B, row_bytes, pr.N, pr.L, k.tile_n / 4, false)) {
        plan->map_bh_ptr = nullptr;
        return BSG_ERR_CUDA;
      }
      plan->map_bh_ptr = B;
    }
    const int chunks = plan->kind == kKindF8F6F4 ? 1 : (plan->kind == kKindF4x4X ? 4 : 2);
    const int k_atoms = chunks * plan->kslices;
    const int sfb_atoms = k.tile_n % 128 == 0 ? (k.tile_n + 127) / 128 : (k.tile_n + 127) / 128 + 1;
    if (plan->map_sfa_ptr != SFA) {
      if (!encode_scales(&plan->map_sfa, SFA, k.t_k, k.t_m, pr.L, k_atoms, 1)) {
        plan->map_sfa_ptr = nullptr;
        return BSG_ERR_CUDA;
      }
      plan->map_sfa_ptr = SFA;
    }
    if (plan->map_sfb_ptr != SFB) {
      if (!encode_scales(&plan->map_sfb, SFB, k.t_k, k.t_n, pr.L, k_atoms, sfb_atoms)) {
        plan->map_sfb_ptr = nullptr;
        return BSG_ERR_CUDA;
      }
      plan->map_sfb_ptr = SFB;
    }
    ma = plan->map_a;
    mb = plan->map_b;
    mbh = k.full_units < k.num_units ? plan->map_bh : plan->map_b;
    msfa = plan->map_sfa;
    msfb = plan->map_sfb;
  }
  void* args[6] = {&ma, &mb, &mbh, &msfa, &msfb, &k};
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(launch_grid(plan, k));
  const void* const fn = k.ks_tiles ? plan->kernel_ks : plan->kernel;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(plan->smem_bytes);
  cfg.stream = static_cast<cudaStream_t>(stream);
  if (plan->cluster_m > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = plan->cluster_m;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  return BSG_OK;
}

// ---------------------------------------------------------------------------
// bsg_run_noalloc: the same launch as bsg_run, with the workspace taken from a
// fixed device array of this library instead of caller memory.  For callers
// that cannot allocate device memory at all (no allocator of their own, or a
// context in which cudaMalloc is not allowed).

// The fixed array: the words every run needs.  A plan whose fastest form
// needs more (the K halves' partial sums) runs the form a small workspace
// gets, as bsg_run does with one.
static constexpr size_t kNoAllocScratchBytes = 4096;
static_assert(kWorkspaceBytes <= kNoAllocScratchBytes, "every plan runs on the fixed array");

// Loaded (zero, having no initialiser) on every GPU that loads this library,
// held until exit.  Host code must not hand this name to a kernel: on the
// host it is only a stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static constexpr int kNoAllocMaxDevices = 64;
static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (the first call on a device).  Nothing is written here: the array
// is zero when the module loads, and every call clears the words a run
// reads on its own stream.
static bsg_status noalloc_scratch(int device, void** out) {
  if (device < 0 || device >= kNoAllocMaxDevices) return BSG_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return BSG_ERR_CUDA;
    }
    g_noalloc_ptr[device] = ptr;
  }
  *out = g_noalloc_ptr[device];
  return BSG_OK;
}

bsg_status bsg_run_noalloc(const bsg_plan* plan, const void* A, const void* B, const void* SFA,
                           const void* SFB, void* C, float* amax, void* stream) {
  if (!plan) return BSG_ERR_INVALID_ARG;
  // the checks bsg_run makes, before the array is looked up or cleared, so
  // that a bad pointer or the wrong current device touches no device state
  bsg_status st = check_run_args(plan, A, B, SFA, SFB, C, amax);
  if (st != BSG_OK) return st;
  void* scratch = nullptr;
  st = noalloc_scratch(plan->device, &scratch);
  if (st != BSG_OK) return st;
  // the array keeps the previous call's words: clear the Amax slot, the
  // arrival counter and the error word before this launch
  if (cudaMemsetAsync(scratch, 0, 16, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  return bsg_run(plan, A, B, SFA, SFB, C, amax, scratch, kNoAllocScratchBytes, stream);
}

bsg_status bsg_run_host(const bsg_plan* plan, const void* hA, const void* hB, const void* hSFA,
                        const void* hSFB, void* hC, float* h_amax, const bsg_device_buffers* dev,
                        void* stream) {
  if (!plan || !hA || !hB || !hSFA || !hSFB || !hC || !h_amax || !dev) return BSG_ERR_INVALID_ARG;
  const bsg_problem& p = plan->prob;
  const bool fp4 = p.a_dtype == BSG_E2M1;
  const size_t a_bytes = static_cast<size_t>(p.L * p.M) * (fp4 ? p.K / 2 : p.K);
  const size_t b_bytes = static_cast<size_t>(p.L * p.N) * (fp4 ? p.K / 2 : p.K);
  const size_t sfa_bytes = static_cast<size_t>(p.L * plan->base.t_m * plan->base.t_k) * kAtomBytes;
  const size_t sfb_bytes = static_cast<size_t>(p.L * plan->base.t_n * plan->base.t_k) * kAtomBytes;
  const size_t c_bytes = static_cast<size_t>(p.L * p.M * c_extent_bytes(p.N, p.c_dtype));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!dev->A || !dev->B || !dev->SFA || !dev->SFB || !dev->C || !dev->amax)
    return BSG_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(dev->A, hA, a_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dev->B, hB, b_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dev->SFA, hSFA, sfa_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dev->SFB, hSFB, sfb_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  const bsg_status st = bsg_run(plan, dev->A, dev->B, dev->SFA, dev->SFB, dev->C, dev->amax,
                                dev->workspace, dev->ws_bytes, stream);
  if (st != BSG_OK) return st;
  if (cudaMemcpyAsync(hC, dev->C, c_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(h_amax, dev->amax, sizeof(float), cudaMemcpyDeviceToHost, s) != cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  return BSG_OK;
}

bsg_status bsg_check_device_status(const bsg_plan* plan, void* ws, void* stream) {
  if (!plan || !ws) return BSG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t words[2] = {0, 0};
  // read and clear the error words on the caller's stream, so that the
  // clear is ordered before the next launch there (a non-blocking stream
  // does not wait for the legacy default stream)
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyAsync(words, static_cast<uint8_t*>(ws) + 8, sizeof(words), cudaMemcpyDeviceToHost,
                      s) != cudaSuccess ||
      cudaMemsetAsync(static_cast<uint8_t*>(ws) + 8, 0, sizeof(words), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  if (words[0] & kErrTimeout) {
    if (std::getenv("BSG_LOG"))
      std::fprintf(stderr, "[bsgemm] device wait timed out (site %u)\n", words[1]);
    return BSG_ERR_DEVICE_TIMEOUT;
  }
  return BSG_OK;
}

bsg_status bsg_plan_describe(const bsg_plan* plan, bsg_plan_info* info) {
  if (!plan || !info) return BSG_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->tile_m = kTileM;
  info->tile_n = plan->base.tile_n;
  info->tile_k_bytes = kStageKBytes * plan->kslices;
  info->stages = plan->base.stages;
  info->grid = plan->grid;
  info->threads = kThreads;
  info->smem_bytes = plan->smem_bytes;
  info->num_tiles = plan->base.num_tiles;
  info->mma_kind = plan->kind;
  info->cluster_m = plan->cluster_m;
  info->half_tiles = plan->half_tiles;
  info->k_split_tiles = plan->ks_tiles;
  std::snprintf(info->kernel_name, sizeof(info->kernel_name), "bsg_gemm_amax_kernel");
  return BSG_OK;
}

void bsg_plan_destroy(bsg_plan* plan) { delete plan; }

}  // extern "C"
