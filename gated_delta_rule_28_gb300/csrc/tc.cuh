// Blackwell (sm_103a) tensor-core building blocks in inline PTX: mbarriers
// with bounded waits, tensor-memory allocation and loads, and tcgen05.mma
// with shared-memory operand descriptors.
//
// Operand layout: bf16 tiles with the 128-byte swizzle. A tile holds rows of
// 64 bf16 (128 bytes); rows come in 8-row, 1024-byte atoms; inside an atom the
// 16-byte chunk index of an element is XORed with (row mod 8). Tiles start on
// 1024-byte boundaries. K-major: a row is one M (or N) index, 64 along K; wider
// K is stored as consecutive 64-wide K-blocks. MN-major: a row is one K index,
// 64 along M (or N) -- the natural layout of a row-major matrix read
// transposed, so that token-major tiles serve as either operand unchanged.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of element (row, k) (k < 64) inside a swizzled K-major tile
__device__ __forceinline__ uint32_t sw128_offset(int row, int k) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((k >> 3) ^ (row & 7)) & 7) << 4) +
                    ((k & 7) << 1));
}

// ---------------------------------------------------------------------------
// mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after `limit` polls (each poll itself blocks for a
// short hardware-defined window) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
#pragma unroll 1
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ---------------------------------------------------------------------------
// tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
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
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// make generic-proxy shared-memory writes visible to the tensor core
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns per thread
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
  uint32_t x[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]),
        "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]),
        "=r"(x[14]), "=r"(x[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = __uint_as_float(x[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// descriptors
// shared-memory operand descriptor: K-major, 128-byte swizzle, 1024-byte atoms
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                   // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024u >> 4) << 32;        // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;                   // descriptor version
  d |= (uint64_t)2 << 61;                   // 128-byte swizzle
  return d;
}

// shared-memory operand descriptor: MN-major, 128-byte swizzle. Each 128-byte row holds 64
// consecutive M (or N) elements of one K index; 8-row atoms of 1024 bytes follow each other
// along K; the next 64 elements along M (N) start `lbo` bytes further on.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);      // start address
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;   // leading byte offset: next 64 along M / N
  d |= (uint64_t)(1024u >> 4) << 32;             // stride byte offset: next 8 rows along K
  d |= (uint64_t)1 << 46;                        // descriptor version
  d |= (uint64_t)2 << 61;                        // 128-byte swizzle
  return d;
}

// instruction descriptor of kind::f16: bf16 x bf16 -> f32; A and B K-major unless a_mn / b_mn
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool negate_a = false, bool a_mn = false,
                                                  bool b_mn = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((negate_a ? 1u : 0u) << 13) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One operand of mma_ops_w: a swizzled tile at `addr`. K-major: 64-wide K-blocks `step` bytes
// apart (a 16-element K step moves 32 bytes inside the block). MN-major: K rows of 128 bytes
// (a 16-element K step moves 2048 bytes), `step` = bytes to the next 64 along M / N.
struct Opnd {
  uint32_t addr, step;
  bool mn;
};
__device__ __forceinline__ Opnd kmaj(uint32_t addr, uint32_t kb) { return Opnd{addr, kb, false}; }
__device__ __forceinline__ Opnd mnmaj(uint32_t addr, uint32_t lbo) { return Opnd{addr, lbo, true}; }

// ---------------------------------------------------------------------------
// Warp-collective issue: called by all 32 lanes of a warp with warp-uniform
// arguments; one elected lane (the same one every time) issues the operation.
// Issuing from warp-uniform code keeps the descriptors in uniform registers: a
// tcgen05.mma issued from a one-thread branch costs tens of cycles of operand
// moves each, one issued this way about one.
__device__ __forceinline__ void mma_bf16_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint64_t *bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar))
      : "memory");
}
// D[M x N] (+)= A[M x K] B[N x K]^T for K a multiple of 16, either operand K- or MN-major
// (the instruction descriptor must say which, idesc_bf16's a_mn / b_mn); warp-collective;
// one MMA per call (K a multiple of 64 goes through mma_grp_w, below)
__device__ __forceinline__ void mma_ops1_w(uint32_t d_tmem, Opnd A, Opnd B, int K, uint32_t idesc, bool accumulate) {
  const uint64_t a0 = A.mn ? sdesc_sw128_mn(A.addr, A.step) : sdesc_sw128(A.addr);
  const uint64_t b0 = B.mn ? sdesc_sw128_mn(B.addr, B.step) : sdesc_sw128(B.addr);
#pragma unroll
  for (int ks = 0; ks < K / 16; ++ks) {
    const uint32_t ao = A.mn ? (uint32_t)ks * 2048u : (uint32_t)(ks >> 2) * A.step + (uint32_t)(ks & 3) * 32u;
    const uint32_t bo = B.mn ? (uint32_t)ks * 2048u : (uint32_t)(ks >> 2) * B.step + (uint32_t)(ks & 3) * 32u;
    mma_bf16_w(d_tmem, a0 + (ao >> 4), b0 + (bo >> 4), idesc, (accumulate || ks > 0) ? 1u : 0u);
  }
}
// Four MMAs of one K=64 block in one asm statement, one elect. The operand descriptors
// are formed inside from their low words (start address >> 4 and the leading byte
// offset, sdesc_sw128 / sdesc_sw128_mn) and the common high word (1 KB stride between
// 8-row atoms, version, 128-byte swizzle); A advances by AO, B by BO (16-byte units) per
// 16-element K step (K-major: 2, MN-major: 128).
constexpr uint32_t SDESC_HI = (1024u >> 4) | (1u << 14) | (2u << 29);
template <int AO, int BO>
__device__ __forceinline__ void mma4_w(uint32_t d_tmem, uint32_t alo, uint32_t blo, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, q, e;\n .reg .b32 x, y;\n .reg .b64 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 q, 0, 0;\n elect.sync _|e, 0xffffffff;\n"
      " mov.b64 a, {%1, %11};\n mov.b64 b, {%2, %11};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n"
      " add.u32 x, %1, %5;\n add.u32 y, %2, %8;\n mov.b64 a, {x, %11};\n mov.b64 b, {y, %11};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n"
      " add.u32 x, %1, %6;\n add.u32 y, %2, %9;\n mov.b64 a, {x, %11};\n mov.b64 b, {y, %11};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n"
      " add.u32 x, %1, %7;\n add.u32 y, %2, %10;\n mov.b64 a, {x, %11};\n mov.b64 b, {y, %11};\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n}\n" ::"r"(d_tmem),
      "r"(alo), "r"(blo), "r"(idesc), "r"(accumulate), "n"(AO), "n"(2 * AO), "n"(3 * AO), "n"(BO), "n"(2 * BO),
      "n"(3 * BO), "n"(SDESC_HI)
      : "memory");
}
// low descriptor word of an operand (sdesc_sw128 / sdesc_sw128_mn)
__device__ __forceinline__ uint32_t sdesc_lo(Opnd X) {
  return ((X.addr & 0x3FFFFu) >> 4) | ((X.mn ? ((X.step >> 4) & 0x3FFFu) : 1u) << 16);
}
// D (+)= A B^T over K (a multiple of 64) in groups of four MMAs; operands as mma_ops_w. The
// loop over the groups stays rolled: one copy of the issue code per call site (the issuing
// warps' loops run from the instruction cache, and this is most of their code)
__device__ __forceinline__ void mma_grp_w(uint32_t d_tmem, Opnd A, Opnd B, int K, uint32_t idesc, bool accumulate) {
  const uint32_t a0 = sdesc_lo(A), b0 = sdesc_lo(B);
#pragma unroll 1
  for (int g = 0; g < K / 64; ++g) {
    // K block g: K-major operands move to the next 64-wide block (`step` bytes), MN-major
    // ones by 4 x 2048 bytes
    const uint32_t ag = a0 + ((A.mn ? (uint32_t)g * 8192u : (uint32_t)g * A.step) >> 4);
    const uint32_t bg = b0 + ((B.mn ? (uint32_t)g * 8192u : (uint32_t)g * B.step) >> 4);
    const uint32_t acc = (accumulate || g > 0) ? 1u : 0u;
    if (A.mn && B.mn) mma4_w<128, 128>(d_tmem, ag, bg, idesc, acc);
    else if (A.mn) mma4_w<128, 2>(d_tmem, ag, bg, idesc, acc);
    else if (B.mn) mma4_w<2, 128>(d_tmem, ag, bg, idesc, acc);
    else mma4_w<2, 2>(d_tmem, ag, bg, idesc, acc);
  }
}
// D (+)= A B^T: groups of four MMAs when K is a multiple of 64 (smaller code), else one
// MMA per K step
__device__ __forceinline__ void mma_ops_w(uint32_t d_tmem, Opnd A, Opnd B, int K, uint32_t idesc, bool accumulate) {
  if (K % 64 == 0) mma_grp_w(d_tmem, A, B, K, idesc, accumulate);
  else mma_ops1_w(d_tmem, A, B, K, idesc, accumulate);
}
// both operands K-major: consecutive 64-wide K-blocks a_kb / b_kb bytes apart; warp-collective
__device__ __forceinline__ void mma_tiles_w(uint32_t d_tmem, uint32_t a_saddr, uint32_t a_kb, uint32_t b_saddr,
                                            uint32_t b_kb, int K, uint32_t idesc, bool accumulate) {
  mma_ops_w(d_tmem, kmaj(a_saddr, a_kb), kmaj(b_saddr, b_kb), K, idesc, accumulate);
}

// TMA (warp-collective, as above): tensor tiles and plain bulk copies into shared memory,
// completing on an mbarrier armed with the expected byte count. A tile's x coordinate times
// 2 bytes must be a multiple of 16 (every caller passes a multiple of 64 elements); a bulk
// copy wants both addresses 16-byte aligned and a size that is a multiple of 16.
__device__ __forceinline__ void mbar_expect_tx_w(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n}\n" ::"r"(smem_u32(bar)), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_w(uint32_t dst, const void *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n}\n" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_load_w(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n}\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk stores shared -> global (warp-collective, the same elected lane each time, so that
// the one thread that commits a group also waits for it): both addresses 16-byte aligned and
// a size that is a multiple of 16.
__device__ __forceinline__ void bulk_store_w(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n"
      " @e cp.async.bulk.commit_group;\n}\n" ::"l"(reinterpret_cast<uint64_t>(dst)),
      "r"(src), "r"(bytes)
      : "memory");
}
// a tensor tile shared -> global (its box from the map; the 128-byte-swizzled layout in shared
// memory), committed as a bulk group of the elected lane, as bulk_store_w
__device__ __forceinline__ void tma_store_2d_w(const void *map, int x, int y, uint32_t src) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n"
      " @e cp.async.bulk.commit_group;\n}\n" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
// the source of every committed bulk store has been read (it may be rewritten)
__device__ __forceinline__ void bulk_store_wait_read_w() {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n @e cp.async.bulk.wait_group.read 0;\n}\n" ::
          : "memory");
}
// every committed bulk store has completed
__device__ __forceinline__ void bulk_store_wait_w() {
  asm volatile("{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n @e cp.async.bulk.wait_group 0;\n}\n" ::
                   : "memory");
}

}  // namespace tc
}  // namespace gdn
