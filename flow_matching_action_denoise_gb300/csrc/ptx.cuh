// Inline-PTX helpers for sm_103a: mbarrier, TMA bulk tensor copies, tcgen05
// (TMEM allocation, MMA, commit, TMEM loads) and Programmatic Dependent Launch.
// Every wait on an mbarrier is bounded by a wall-clock budget read from
// %globaltimer; callers turn an expired wait into an error-word bit.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace fm {

constexpr uint64_t kWaitBudgetNs = 2000000000ull;   // 2 s: far beyond any legitimate wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- PDL
// Wait until the preceding grid in the stream has completed and its writes are
// visible. Every kernel calls this before touching data an earlier kernel wrote.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid in the stream to be scheduled (its pre-wait prologue runs
// while this grid finishes).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done;
}
// True once the phase with the given parity has completed; false if the budget expired.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns = kWaitBudgetNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > budget_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA
// Asynchronous prefetch of [src, src + bytes) from global memory into L2 (bytes and
// src: multiples of 16); no completion to wait for.
__device__ __forceinline__ void l2_prefetch_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
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
// 2-D tiled load of one box into shared memory; completion is signalled on `bar`
// as transaction bytes. c0 is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// 3-D tiled load (c0 innermost); completion signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Plain bulk copy of `bytes` contiguous bytes (16-byte aligned both sides, size a
// multiple of 16) into shared memory, completion signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation is warp-collective; the allocated base address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// D[tmem] (+)= A[smem desc] x B[smem desc]; kind::f8f6f4 (E4M3 x E4M3) or kind::f16 (BF16 x BF16).
template <bool kFp8>
__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  if constexpr (kFp8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// The same MMA with the A operand read from tensor memory: a_tmem is the TMEM address
// of A's first column (M = 128: row i in lane i, K along the columns, 32-bit cells
// holding two 16-bit or four 8-bit elements).
template <bool kFp8>
__device__ __forceinline__ void tc_mma_ts(uint32_t tmem_d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (kFp8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Each thread of a warp writes 4, 8 or 16 consecutive 32-bit columns of its TMEM lane
// (warp-collective); tmem_wait_st() waits for the warp's stores to be done.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand stored in the canonical
// 128-byte-swizzle layout (rows of 128 bytes, 8-row core groups 1024 bytes apart,
// as a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes it). The tile base must be
// 1024-byte aligned; advancing along K inside the 128-byte row adds to the start.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // bits 0-13: start address >> 4
  d |= static_cast<uint64_t>(0) << 16;                     // bits 16-29: leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;             // bits 32-45: stride byte offset >> 4
  d |= static_cast<uint64_t>(1) << 46;                     // bits 46-48: descriptor version 0b001
  d |= static_cast<uint64_t>(2) << 61;                     // bits 61-63: 128-byte swizzle
  return d;
}

// Instruction descriptor: F32 accumulate, both operands K-major, shape M x N.
// a/b format: E4M3 = 0 under kind::f8f6f4, BF16 = 1 under kind::f16.
__device__ __forceinline__ uint32_t make_idesc(bool fp8, uint32_t mma_m, uint32_t mma_n) {
  const uint32_t fmt = fp8 ? 0u : 1u;
  return (1u << 4)                 // D format F32
         | (fmt << 7)              // A format
         | (fmt << 10)             // B format
         | ((mma_n >> 3) << 17)    // N >> 3
         | ((mma_m >> 4) << 24);   // M >> 4
}

// Instruction descriptor of kind::f16 with f16 A and B (format code 0), fp32 D.
__device__ __forceinline__ uint32_t make_idesc_f16(uint32_t mma_m, uint32_t mma_n) {
  return (1u << 4) | ((mma_n >> 3) << 17) | ((mma_m >> 4) << 24);
}

// Each thread of a warp reads 16 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Each thread of a warp reads 32 consecutive 32-bit columns of its TMEM lane (one load,
// one wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x by the MUFU instruction (approximate, denormal results flushed to zero); the
// attention's probabilities are rounded to bf16 or E4M3 afterwards.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- clusters
// Split cluster barrier: arrive early (relaxed: orders nothing), wait later. Used
// to know every peer CTA has started before writing into its shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// Bulk copy (TMA engine) from this CTA's shared memory to the shared memory of a CTA
// of the cluster; `dst` and `mbar` are shared::cluster addresses in the destination
// CTA, whose mbarrier receives the byte count. Addresses and size: multiples of 16.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "r"(src), "r"(bytes), "r"(mbar)
               : "memory");
}
// Asynchronous 4-byte store into a CTA of the cluster, counted on that CTA's mbarrier
// (shared::cluster addresses).
__device__ __forceinline__ void st_async_f32(uint32_t dst, float a, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(dst), "f"(a),
               "r"(mbar)
               : "memory");
}
// Asynchronous 16-byte store into a CTA of the cluster, counted on that CTA's mbarrier
// (shared::cluster addresses; dst 16-byte aligned).
__device__ __forceinline__ void st_async_v4(uint32_t dst, float a, float b, float c, float d, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(dst), "f"(a), "f"(b), "f"(c), "f"(d), "r"(mbar)
               : "memory");
}
// Transpose of a 4 x 4 block held by the four lanes of an aligned lane group: lane t
// holds row t on entry and column t on exit. Two butterfly exchanges: the off-diagonal
// 2 x 2 blocks swap between lanes t and t ^ 2, then each 2 x 2 block transposes between
// lanes t and t ^ 1. Every lane of the warp must execute it.
__device__ __forceinline__ void transpose4x4(float& x0, float& x1, float& x2, float& x3, int t) {
  const bool hi = (t & 2) != 0;
  float a = hi ? x0 : x2, b = hi ? x1 : x3;
  a = __shfl_xor_sync(0xffffffffu, a, 2);
  b = __shfl_xor_sync(0xffffffffu, b, 2);
  if (hi) {
    x0 = a;
    x1 = b;
  } else {
    x2 = a;
    x3 = b;
  }
  const bool odd = (t & 1) != 0;
  a = odd ? x0 : x1;
  b = odd ? x2 : x3;
  a = __shfl_xor_sync(0xffffffffu, a, 1);
  b = __shfl_xor_sync(0xffffffffu, b, 1);
  if (odd) {
    x0 = a;
    x2 = b;
  } else {
    x1 = a;
    x3 = b;
  }
}
// Asynchronous 8-byte store into a CTA of the cluster, counted on that CTA's mbarrier
// (shared::cluster addresses).
__device__ __forceinline__ void st_async_v2(uint32_t dst, float a, float b, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(dst), "f"(a), "f"(b), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Map a local shared-memory address to the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_dsmem(uint32_t saddr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(saddr), "r"(rank));
  return out;
}

// ---------------------------------------------------------------- timeline (diagnostics)
// When a kernel is given a timeline buffer, thread 0 of each CTA appends one 128-byte
// record: word 0 identifies the CTA (kind | gridDim.x << 8 | grid rows << 20 |
// blockIdx.x << 32 | block row << 44 | SM id << 56), words 1-15 are %globaltimer stamps
// (ns) at points the kernel defines (0 = not reached). Buffer: u32 count, u32 capacity,
// 56 bytes of padding, then the records; records past the capacity are dropped.
constexpr int kTlStamps = 15;
enum TlKind : uint32_t { kTlGemm = 1, kTlAttn = 2, kTlRow = 3, kTlNvfp4 = 4 };

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void tl_record(unsigned long long* tl, uint32_t kind, uint32_t grid_rows, uint32_t row,
                                          const uint64_t* t) {
  unsigned* hdr = reinterpret_cast<unsigned*>(tl);
  const unsigned idx = atomicAdd(hdr, 1u);
  if (idx >= hdr[1]) return;
  unsigned long long* rec = tl + 8 + static_cast<size_t>(idx) * 16;
  rec[0] = static_cast<unsigned long long>(kind) | (static_cast<unsigned long long>(gridDim.x & 0xfff) << 8) |
           (static_cast<unsigned long long>(grid_rows & 0xfff) << 20) |
           (static_cast<unsigned long long>(blockIdx.x & 0xfff) << 32) |
           (static_cast<unsigned long long>(row & 0xfff) << 44) | (static_cast<unsigned long long>(sm_id() & 0xff) << 56);
#pragma unroll
  for (int i = 0; i < kTlStamps; ++i) rec[1 + i] = t[i];
}

}  // namespace fm
