// Inline-PTX wrappers for sm_103a: mbarriers with bounded waits, TMA tile loads
// and stores (cp.async.bulk.tensor, one CTA, no multicast), and the 5th-generation tensor
// core (tcgen05: TMEM allocation, MMA with shared-memory descriptors, commit,
// TMEM loads). Every wait is bounded by a wall-clock budget; a wait that runs
// out records an error in a device status word and returns false so the
// caller can leave cleanly instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdp {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
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

// Wait budget for one phase of one barrier (nanoseconds of wall time): 2 s,
// unless the test hook gdp_debug_wait_fault has set a shorter one.
constexpr uint64_t kWaitBudgetNs = 2000000000ull;
static __device__ unsigned long long g_wait_budget_ns = kWaitBudgetNs;

// Bounded wait for `parity`; on timeout stores `code` into *status (if not
// null) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, int code) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t budget = *const_cast<volatile unsigned long long*>(&g_wait_budget_ns);
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (globaltimer_ns() - t0 > budget) {
      if (status) atomicExch(status, code);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA (tile mode)
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// Tiled bulk store shared -> global (coordinates must be >= 0; the innermost one
// times the element size a multiple of 16 bytes). Completion is tracked by the
// issuing thread's bulk groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk store of this thread has finished reading
// shared memory (READ) or has completed (all writes performed).
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// The same, but the most recent committed group may still be reading.
__device__ __forceinline__ void tma_store_wait_read_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tcgen05.mma).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation is warp-wide (.sync.aligned): call from one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulation (kind::f16).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same MMA with the accumulate flag as an immediate (ACC: add to D).
template <bool ACC>
__device__ __forceinline__ void mma_bf16_i(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "n"(ACC ? 1 : 0)
      : "memory");
}

// NK MMAs along K into one accumulator, D (+)= sum_k A_k B_k, from the base
// descriptors of A_0 and B_0: step k moves A by (k / 4) A_HI + (k % 4) A_LO bytes
// and B by (k / 4) B_HI + (k % 4) B_LO bytes (a 128-byte swizzle atom holds four
// 16-element K steps). The steps are added to the descriptors' address field
// (no carry out of it: shared addresses stay below 256 KB), so each MMA costs one
// 64-bit add per operand instead of building its descriptors from scratch; the
// first MMA overwrites D unless ACC0.
template <int NK, bool ACC0, int A_HI, int A_LO, int B_HI, int B_LO>
__device__ __forceinline__ void mma_run(uint32_t d_tmem, uint64_t a0, uint64_t b0, uint32_t idesc) {
  mma_bf16_i<ACC0>(d_tmem, a0, b0, idesc);
#pragma unroll
  for (int kk = 1; kk < NK; ++kk)
    mma_bf16_i<true>(d_tmem, a0 + (uint64_t)((((kk >> 2) * A_HI) + (kk & 3) * A_LO) >> 4),
                     b0 + (uint64_t)((((kk >> 2) * B_HI) + (kk & 3) * B_LO) >> 4), idesc);
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, dense.
// a_mn / b_mn select MN-major (1) instead of K-major (0) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                      // D format: f32
         | (1u << 7)                    // A format: bf16
         | (1u << 10)                   // B format: bf16
         | ((a_mn ? 1u : 0u) << 15)     // A major
         | ((b_mn ? 1u : 0u) << 16)     // B major
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B). lbo/sbo in bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Shared-memory matrix descriptor, 64-byte swizzle: 64-byte rows, 8-row groups
// of 512 bytes, 16-byte chunk j of row r stored at chunk j ^ ((r >> 1) & 3).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (4ull << 61);
}

// Byte offset of 16-byte chunk j (0..3) of row r in a 64B-swizzled tile.
__device__ __forceinline__ uint32_t sw64_chunk(uint32_t r, uint32_t j) {
  return r * 64u + ((j ^ ((r >> 1) & 3u)) << 4);
}

// TMEM -> registers: the calling warp reads its 32 lanes (lane base = 32 * (warp % 4),
// encoded in taddr bits 31:16), 16 or 32 consecutive 32-bit columns each.
#define GDP_TMEM_LD8(taddr, r)                                                             \
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"   \
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),  \
                 "=r"(r[6]), "=r"(r[7])                                                   \
               : "r"(taddr))

#define GDP_TMEM_LD16(taddr, r)                                                            \
  asm volatile(                                                                           \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "                                           \
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"                   \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),           \
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),         \
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])                                \
      : "r"(taddr))

#define GDP_TMEM_LD32(taddr, r)                                                             \
  asm volatile(                                                                            \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "                                            \
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"                            \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"           \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),            \
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),          \
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),      \
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),      \
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),      \
        "=r"(r[30]), "=r"(r[31])                                                           \
      : "r"(taddr))

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Byte offset of element (row, col16) inside a 128B-swizzled tile whose rows are
// 128 bytes: 16-byte chunk index col16 (0..7) is XOR-ed with row % 8.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t byte_in_row) {
  const uint32_t chunk = (byte_in_row >> 4) ^ (row & 7u);
  return row * 128u + (chunk << 4) + (byte_in_row & 15u);
}

}  // namespace ptx
}  // namespace gdp
