// Fifth-generation tensor core (tcgen05) building blocks for sm_103a, in inline
// PTX: tensor-memory allocation, shared-memory matrix descriptors for the
// no-swizzle K-major layout, the MMA issued by one thread with its fp32
// accumulator in tensor memory, completion through an mbarrier, and the
// 32-lane × 32-bit tensor-memory loads of the epilogue.
//
// Operand layout in shared memory (no swizzle, K-major): a tile of R rows × K
// columns of 16-bit elements is stored as 8 × 8 "core matrices" of 128
// contiguous bytes (8 rows of 16 bytes).  Core matrix (row group rg, column
// group kg) sits at byte ((kg · R/8) + rg) · 128, row r % 8 at 16 · (r % 8),
// column k % 8 at 2 · (k % 8).  In the descriptor the leading byte offset is
// the distance between column groups (R/8 · 128) and the stride byte offset the
// distance between row groups (128).
#pragma once

#include <cstdint>

namespace ssm {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of element (r, k) of an R-row K-major core-matrix tile
__host__ __device__ constexpr uint32_t kmajor_offset(int R, int r, int k) {
  return (uint32_t)((((k >> 3) * (R >> 3)) + (r >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (all >> 4), descriptor version 1 (bits 46-47), no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// descriptor of the K = 16 slice kk of an R-row K-major tile at `base`
__device__ __forceinline__ uint64_t kslice_desc(uint32_t base, int R, int kk) {
  return smem_desc(base + (uint32_t)(kk * 2 * (R / 8) * 128), (uint32_t)((R / 8) * 128), 128u);
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator, both
// operands K-major, M × N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with either operand MN-major (bit 15: A, bit 16: B).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_major(int M, int N, bool a_mn, bool b_mn) {
  return idesc_bf16_f32(M, N) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16);
}

// 128-byte swizzle (layout type 2 in bits 61-63): rows of 128 bytes, the 16-byte
// chunk j of row r stored at chunk j ^ (r % 8), 8-row groups of 1024 bytes — the
// layout a tensor copy with CU_TENSOR_MAP_SWIZZLE_128B writes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return smem_desc(addr, lbo, sbo) | (2ull << 61);
}
// K-major, 128-byte swizzle: R rows × 128 K stored as two column blocks (K 0..63,
// 64..127) of R × 128 bytes; the K = 16 slice kk starts 32 bytes into its block's rows.
__device__ __forceinline__ uint64_t sw128_kslice_desc(uint32_t base, int R, int kk) {
  return sw128_desc(base + (uint32_t)((kk >> 2) * R * 128 + (kk & 3) * 32), 16u, 1024u);
}
// MN-major, 128-byte swizzle: K rows of 128 bytes (64 elements of M or N) per atom
// column, atom columns `atom_stride` bytes apart; the K = 16 slice kk is 16 rows in.
__device__ __forceinline__ uint64_t sw128_mn_kslice_desc(uint32_t base, uint32_t atom_stride, int kk) {
  return sw128_desc(base + (uint32_t)(kk * 2048), atom_stride, 1024u);
}

// MN-major operands (no swizzle): the core matrix is 8 rows along K, each 16
// bytes (8 elements) along M or N.  A tile with 16 groups of 8 along K, stored
// with core matrix (mn group i, k group j) at byte (i · 16 + j) · 128 — the same
// bytes as kmajor_offset(128, k, mn) — has K-direction neighbours 128 bytes apart
// (leading byte offset) and M/N-direction neighbours 2048 bytes apart (stride
// byte offset); its K = 16 slice kk starts at byte 256 · kk.
__device__ __forceinline__ uint64_t mn_kslice_desc(uint32_t base, int kk) {
  return smem_desc(base + (uint32_t)(kk * 256), 128u, 2048u);
}

// D[tmem] (+)= A · Bᵀ for one K = 16 slice; issued by a single thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}
// the mbarrier gets one arrival once every MMA issued so far by this thread is complete
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
               : "memory");
}

// tensor memory: allocation and release by one whole warp
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes made visible to the tensor core's reads
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's lane (warp w reads lanes 32w..32w+31)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
// 16 consecutive fp32 columns of this thread's lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ uint32_t tmem_lane_addr(uint32_t base, int lane0, int col) {
  return base + ((uint32_t)lane0 << 16) + (uint32_t)col;
}

// mbarrier with a single expected arrival
__device__ __forceinline__ void mbar_init1(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// the same, but the thread may sleep until the phase completes, at most `hint_ns`
// nanoseconds, instead of returning at once: a waiting warp issues no instructions
__device__ __forceinline__ bool mbar_test_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

}  // namespace tc
}  // namespace ssm
