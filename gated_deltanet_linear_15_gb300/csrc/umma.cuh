// Blackwell (sm_100 family) primitives written as inline PTX: tensor memory
// (TMEM) allocation, tcgen05.mma with shared-memory operand descriptors,
// tcgen05.ld/st, mbarriers with bounded waits, and TMA tile loads.
//
// Shared-memory operand layout used throughout: 128-byte swizzle.  A tile of R
// rows x 64 sixteen-bit elements occupies R * 128 bytes, row r at r * 128, and
// the 16-byte chunk c of row r is stored at chunk position c ^ (r % 8) (tile
// base 1024-byte aligned).  TMA with CU_TENSOR_MAP_SWIZZLE_128B writes exactly
// this layout, and the MMA reads it through descriptors:
//  - K-major operand (rows = M or N, the 64 elements of a row run along K):
//    stride between 8-row groups (SBO) = 1024 bytes; a K step of 16 elements
//    moves the start address by 32 bytes inside the 128-byte row.
//  - MN-major operand (rows = K, the 64 elements of a row run along M or N):
//    SBO = 1024 bytes between 8-row groups along K, LBO = stride between
//    64-wide blocks along M/N; a K step of 16 moves the start by 2 * SBO.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace gdn {
namespace umma {

// ------------------------------------------------------------------ swizzle
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col_elem16) {
  // byte offset of 16-bit element (row, col) in a 128B-swizzled [rows][64] tile
  const uint32_t chunk = (col_elem16 >> 3) ^ (row & 7);
  return row * 128u + chunk * 16u + (col_elem16 & 7u) * 2u;
}

// ------------------------------------------------------------------ fragments of [rows][64] tiles
// byte offset of the 16-byte chunk holding columns [cb, cb + 8) of row r in a swizzled tile
__device__ __forceinline__ uint32_t chunk_off(int r, int cb) { return r * 128 + ((((cb & 63) >> 3) ^ (r & 7)) << 4); }

// Transposing read-outs of a [feature lanes][token columns] accumulator (o, dv, dq, dk): warp (wq, wg) reads
// features 32 wq + ls .. + 15 (ls = 0, 16) and tokens c0 .. c0 + 15 as fragments (tmem_ld_frag2), so value
// 2m + e of lane t is feature 32 wq + ls + 8 (m & 1) + t/4, token c0 + 8 (m >> 1) + 2 (t%4) + e; the four
// 8 x 8 matrices m move between those fragments and a token-major [token][feature] tile (feature halves
// `blk` bytes apart, 128-byte swizzled rows) by one ldmatrix / stmatrix .trans, for which lane t addresses
// the 16 bytes of token c0 + 8 ((t/8) >> 1) + t%8, features from 32 wq + ls + 8 ((t/8) & 1).
__device__ __forceinline__ uint32_t frag_addr(const uint8_t *base, int blk, int wq, int ls, int c0, int lane) {
  const int m = lane >> 3;
  const int tk = c0 + 8 * (m >> 1) + (lane & 7);
  const int fs = 32 * wq + ls + 8 * (m & 1);
  return smem_u32(base + (fs >> 6) * blk + chunk_off(tk, fs));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&b);
}
__device__ __forceinline__ float2 unpack_f16(uint32_t r) { return __half22float2(*reinterpret_cast<const __half2 *>(&r)); }
// a per-token factor at this lane's four tokens c0 + 2 (t%4) + {0, 1, 8, 9} (16-byte aligned arrays)
__device__ __forceinline__ void tok4(const float *p, int ta, float (&v)[4]) {
  const float2 a = *reinterpret_cast<const float2 *>(p + ta), b = *reinterpret_cast<const float2 *>(p + ta + 8);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}

// ------------------------------------------------------------------ descriptors
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for the sm_100 family
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16 with fp16 A/B and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major, bool neg_a = false) {
  return (1u << 4)                              // D format: f32
         | (0u << 7) | (0u << 10)               // A, B format: f16
         | ((neg_a ? 1u : 0u) << 13)            // negate A
         | ((a_mn_major ? 1u : 0u) << 15)       // A major-ness (0: K-major)
         | ((b_mn_major ? 1u : 0u) << 16)       // B major-ness
         | ((uint32_t)(N >> 3) << 17)           // N / 8
         | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// ------------------------------------------------------------------ TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_dst), "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// A shared-memory operand descriptor as its two 32-bit words.  The start address (>> 4) is the low 14 bits of
// `lo` and every address of the CTA's shared memory window is below 256 KB, so moving the start by a byte
// offset (a K step, another tile) is one add to `lo`: built once, stepped in the issue loops.
struct SDesc {
  uint32_t lo, hi;
};
__device__ __forceinline__ SDesc sdesc_s(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  const uint64_t d = sdesc(saddr, lbo_bytes, sbo_bytes);
  return SDesc{(uint32_t)d, (uint32_t)(d >> 32)};
}
__device__ __forceinline__ SDesc operator+(SDesc d, uint32_t bytes) { return SDesc{d.lo + (bytes >> 4), d.hi}; }
// D[tmem] (+)= A * B with descriptors in that form (accumulate: 0 overwrites D)
__device__ __forceinline__ void mma_f16s(uint32_t d_tmem, SDesc a, SDesc b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .b64 da, db;\n"
      ".reg .pred p;\n"
      "mov.b64 da, {%1, %2};\n"
      "mov.b64 db, {%3, %4};\n"
      "setp.ne.b32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(accumulate));
}
// arrive on an mbarrier once all previously issued MMAs of this thread completed
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
               : "memory");
}

// 32 lanes x 32 columns of fp32: thread t of the warp gets lane (32*(warp%4) + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 8 columns of fp32 (same lane rule as tmem_ld32)
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// two 8-column loads (32 lanes each, same lane rule), one wait
__device__ __forceinline__ void tmem_ld8x2(uint32_t ta, float (&va)[8], uint32_t tb, float (&vb)[8]) {
  uint32_t ra[8], rb[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(ra[0]), "=r"(ra[1]), "=r"(ra[2]), "=r"(ra[3]), "=r"(ra[4]), "=r"(ra[5]), "=r"(ra[6]), "=r"(ra[7])
               : "r"(ta));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(rb[0]), "=r"(rb[1]), "=r"(rb[2]), "=r"(rb[3]), "=r"(rb[4]), "=r"(rb[5]), "=r"(rb[6]), "=r"(rb[7])
               : "r"(tb));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    va[i] = __uint_as_float(ra[i]);
    vb[i] = __uint_as_float(rb[i]);
  }
}
// 32 lanes x 16 columns of fp32 without waiting: call tmem_wait_ld() before using v
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  tmem_ld16_nw(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// two 16-column loads, one wait
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, float (&va)[16], uint32_t tb, float (&vb)[16]) {
  uint32_t ra[16], rb[16];
  tmem_ld16_nw(ta, ra);
  tmem_ld16_nw(tb, rb);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    va[i] = __uint_as_float(ra[i]);
    vb[i] = __uint_as_float(rb[i]);
  }
}
// Fragment loads for transposing read-outs: 16 lanes x 16 columns of fp32 per warp (two 16x256b blocks),
// the accumulator fragment of a 16 x 8 MMA tile twice.  With lane base L and column base C (taddr), thread t
// holds v[4x + 0..1] = lane L + t/4, columns C + 8x + 2(t%4) + {0, 1} and v[4x + 2..3] = lane L + 8 + t/4,
// the same columns (x = 0, 1).  Two loads, one wait.
__device__ __forceinline__ void tmem_ld_frag2(uint32_t ta, float (&va)[8], uint32_t tb, float (&vb)[8]) {
  uint32_t ra[8], rb[8];
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(ra[0]), "=r"(ra[1]), "=r"(ra[2]), "=r"(ra[3]), "=r"(ra[4]), "=r"(ra[5]), "=r"(ra[6]), "=r"(ra[7])
               : "r"(ta));
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(rb[0]), "=r"(rb[1]), "=r"(rb[2]), "=r"(rb[3]), "=r"(rb[4]), "=r"(rb[5]), "=r"(rb[6]), "=r"(rb[7])
               : "r"(tb));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    va[i] = __uint_as_float(ra[i]);
    vb[i] = __uint_as_float(rb[i]);
  }
}
// one fragment load (same layout as tmem_ld_frag2), then wait
__device__ __forceinline__ void tmem_ld_frag1(uint32_t ta, float (&va)[8]) {
  uint32_t ra[8];
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(ra[0]), "=r"(ra[1]), "=r"(ra[2]), "=r"(ra[3]), "=r"(ra[4]), "=r"(ra[5]), "=r"(ra[6]), "=r"(ra[7])
               : "r"(ta));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) va[i] = __uint_as_float(ra[i]);
}
// Four 8 x 8 b16 matrices between fragments and shared memory, not transposed: register i holds row t/4,
// columns 2(t%4) and 2(t%4) + 1 (low half first) of matrix i; thread t gives the address of row t%8 of
// matrix t/8 (16 bytes).
__device__ __forceinline__ void stmatrix_x4(uint32_t saddr, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(saddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t saddr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr)
               : "memory");
}
// Four 8 x 8 b16 matrices between fragments and shared memory, transposed: register i holds fragment row
// t/4, columns 2(t%4) and 2(t%4) + 1 (low half first) of matrix i; thread t gives the address of row t%8 of
// matrix t/8, and that 16-byte row holds column t%8 of the fragment.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(saddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t saddr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr)
               : "memory");
}
// 32 lanes x 32 columns of fp32 into TMEM; tmem_st32_issue leaves the store in flight (tmem_wait_st completes
// every store this thread issued), tmem_st32 waits for it
__device__ __forceinline__ void tmem_st32_issue(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  tmem_st32_issue(taddr, v);
  tmem_wait_st();
}

// ------------------------------------------------------------------ mbarriers
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar), "r"(count));
}
// retire an mbarrier whose phases are all complete, so that its word can be initialised again
__device__ __forceinline__ void mbar_inval(uint32_t mbar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(mbar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mbar), "r"(bytes) : "memory");
}
// raise the transaction bytes the current phase waits for, without arriving (the phase cannot complete before
// its arrival, so loads issued in parts expect their bytes this way and the last part arrives)
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(mbar) : "memory");
}
// Named barriers over part of a CTA (ID and thread count are compile-time: a multiple of 32).  sync
// waits for `N` arrivals; arrive counts the calling warp without waiting.
template <int ID, int N>
__device__ __forceinline__ void named_bar_sync() {
  asm volatile("bar.sync %0, %1;\n" ::"n"(ID), "n"(N) : "memory");
}
template <int ID, int N>
__device__ __forceinline__ void named_bar_arrive() {
  asm volatile("bar.arrive %0, %1;\n" ::"n"(ID), "n"(N) : "memory");
}
// Wait for the phase with the given parity to complete.  Bounded: after
// `limit` polls it records `code` in *err and returns false (never hangs).
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, int *err, int code,
                                          uint32_t limit = (1u << 26)) {
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  if (err) atomicOr(err, code);
  return false;
}

// Test hook for the bounded waits: wait on a fresh barrier that nothing arrives at, with a short
// bound, so the wait expires and records `code` in *err.  Called by thread 0 before the kernel has
// allocated TMEM or issued any copy or product; the caller then returns.
__device__ __forceinline__ void debug_expire_wait(uint64_t *bar, int *err, int code) {
  mbar_init(smem_u32(bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  mbar_wait(smem_u32(bar), 0, err, code, 1024);
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_3d(uint32_t smem_dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
      : "memory");
}
// contiguous global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completing on an mbarrier's transaction count
__device__ __forceinline__ void bulk_load(uint32_t smem_dst, const void *gsrc, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_dst),
               "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(mbar)
               : "memory");
}
// shared -> global tile store (bulk-group completion); the source must have been written before a
// fence.proxy.async.shared::cta and a barrier, and stays untouched until tma_store_wait_read()
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, int x, int y, int z, uint32_t smem_src) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(smem_src)
               : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// the issuing thread's stores have finished reading shared memory
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// the same for all but the most recent store group (which may still be reading its source)
__device__ __forceinline__ void tma_store_wait_read_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory");
}
// the issuing thread's stores are complete
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace umma
}  // namespace gdn
