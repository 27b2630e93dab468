// Thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM allocation, MMA, commit, loads/stores) and the shared-memory /
// instruction descriptors the tcgen05 MMA consumes. Written from the public
// PTX ISA description of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace aa {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
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

// Bounded wait for the phase with the given parity to complete. Returns false
// (and records `site` in the device error word) once `limit_ns` has passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                          int32_t* err, int32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 >= limit_ns) {
      atomicCAS(err, 0, site);
      return false;
    }
  }
}

// Named barrier over `nthreads` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

// ------------------------------------------------------------------ fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled load of box {c, h, t} into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t c,
                                            int32_t h, int32_t t) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c), "r"(h), "r"(t)
      : "memory");
}

// 3-D tiled reduce-add of a shared-memory box into global memory (fp32 add),
// tracked by the issuing thread's bulk group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, const void* src, int32_t c, int32_t h,
                                                  int32_t t) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c), "r"(h), "r"(t)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until all committed bulk groups of this thread have finished reading
// their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// ------------------------------------------------------------------ tcgen05
// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to *slot. Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// tcgen05.mma kind::f16 (bf16 in, fp32 accumulate): D[tmem] (+)= A * B^T with
// A from shared memory (a descriptor) or from TMEM (M rows = TMEM lanes, two
// bf16 K-elements per 32-bit column, K-major) and B from shared memory.
// Eight (or four) MMAs of one product, issued from a single asm block: the
// k-th (k > 0) adds compile-time offsets to the first step's descriptors (in
// 16-byte units, i.e. straight into the descriptors' address fields; no carry
// leaves them since every operand lies inside the 256 KB shared window) or to
// the A operand's TMEM column. Issued one asm statement at a time, an MMA
// holds its warp about twice as long as the tensor core needs for an N = 128
// step; one block lets the issues run back to back. The first MMA accumulates
// only if `accumulate` != 0, the others always.
#define AA_MMA_SS_STEP(ao, bo)                                                            \
  "add.s64 ra, %1, " #ao ";\n\tadd.s64 rb, %2, " #bo ";\n\t"                          \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
#define AA_MMA_TS_STEP(ao, bo)                                                            \
  "add.u32 rt, %1, " #ao ";\n\tadd.s64 rb, %2, " #bo ";\n\t"                          \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [rt], rb, %3, t;\n\t"
#define AA_MMA_PROLOGUE                                                                   \
  "{\n\t.reg .pred p, t;\n\t.reg .b64 ra, rb;\n\t.reg .b32 rt;\n\t"                 \
  "setp.ne.b32 p, %4, 0;\n\tsetp.eq.u32 t, %4, %4;\n\t"

// A and B K-major with the 128-byte swizzle, 64 K-elements per 16 KB block:
// K-steps 0-3 advance 32 bytes inside a block, steps 4-7 start the next block.
__device__ __forceinline__ void mma8_ss_kk(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               AA_MMA_SS_STEP(2, 2) AA_MMA_SS_STEP(4, 4) AA_MMA_SS_STEP(6, 6) AA_MMA_SS_STEP(1024, 1024)
               AA_MMA_SS_STEP(1026, 1026) AA_MMA_SS_STEP(1028, 1028) AA_MMA_SS_STEP(1030, 1030) "}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// Four K-steps of the same layout (one 64-element block: D = 64 products).
__device__ __forceinline__ void mma4_ss_kk(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               AA_MMA_SS_STEP(2, 2) AA_MMA_SS_STEP(4, 4) AA_MMA_SS_STEP(6, 6) "}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// A K-major with the 128-byte swizzle (as above), B MN-major: each K-step
// (16 rows of 128 bytes) advances B by 2048 bytes.
__device__ __forceinline__ void mma8_ss_km(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               AA_MMA_SS_STEP(2, 128) AA_MMA_SS_STEP(4, 256) AA_MMA_SS_STEP(6, 384) AA_MMA_SS_STEP(1024, 512)
               AA_MMA_SS_STEP(1026, 640) AA_MMA_SS_STEP(1028, 768) AA_MMA_SS_STEP(1030, 896) "}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// A and B MN-major: both advance 2048 bytes per K-step.
__device__ __forceinline__ void mma8_ss_mm(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               AA_MMA_SS_STEP(128, 128) AA_MMA_SS_STEP(256, 256) AA_MMA_SS_STEP(384, 384) AA_MMA_SS_STEP(512, 512)
               AA_MMA_SS_STEP(640, 640) AA_MMA_SS_STEP(768, 768) AA_MMA_SS_STEP(896, 896) "}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// A from TMEM (two bf16 K-elements per column, 8 columns per K-step),
// B MN-major (2048 bytes per K-step). `a` is the first step's TMEM address;
// steps 0-3 take columns a + 8k, steps 4-7 columns a + 64 + 8(k - 4): the two
// 32-column halves that two 64-column groups of a 128-wide operand use.
__device__ __forceinline__ void mma8_ts_split(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               AA_MMA_TS_STEP(8, 128) AA_MMA_TS_STEP(16, 256) AA_MMA_TS_STEP(24, 384) AA_MMA_TS_STEP(64, 512)
               AA_MMA_TS_STEP(72, 640) AA_MMA_TS_STEP(80, 768) AA_MMA_TS_STEP(88, 896) "}"
               ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// A from TMEM, consecutive: step k takes columns a + 8k; B MN-major.
__device__ __forceinline__ void mma8_ts_seq(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               AA_MMA_TS_STEP(8, 128) AA_MMA_TS_STEP(16, 256) AA_MMA_TS_STEP(24, 384) AA_MMA_TS_STEP(32, 512)
               AA_MMA_TS_STEP(40, 640) AA_MMA_TS_STEP(48, 768) AA_MMA_TS_STEP(56, 896) "}"
               ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// Half of an eight-step product whose K runs over two 64-wide halves (query
// columns 0-63 and 64-127): part 0 takes K-steps 0, 1, 4, 5 (columns 0-31 and
// 64-95), part 1 K-steps 2, 3, 6, 7. A from TMEM at columns a + 8k' (k' the
// step's column offset within the 128-wide operand), B MN-major.
__device__ __forceinline__ void mma4_ts_part0(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               AA_MMA_TS_STEP(8, 128) AA_MMA_TS_STEP(64, 512) AA_MMA_TS_STEP(72, 640) "}"
               ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma4_ts_part1(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "add.u32 rt, %1, 16;\n\tadd.s64 rb, %2, 256;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [rt], rb, %3, p;\n\t"
               AA_MMA_TS_STEP(24, 384) AA_MMA_TS_STEP(80, 768) AA_MMA_TS_STEP(88, 896) "}"
               ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// The same split for A K-major with the 128-byte swizzle (two 64-column
// blocks) and B MN-major.
__device__ __forceinline__ void mma4_ss_part0(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               AA_MMA_SS_STEP(2, 128) AA_MMA_SS_STEP(1024, 512) AA_MMA_SS_STEP(1026, 640) "}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma4_ss_part1(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(AA_MMA_PROLOGUE
               "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 256;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, p;\n\t"
               AA_MMA_SS_STEP(6, 384) AA_MMA_SS_STEP(1028, 768) AA_MMA_SS_STEP(1030, 896) "}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// Arrive once on `bar` when all previously issued MMAs of this thread finish.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Each thread of the warp reads 32 consecutive fp32 columns of its own lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Each thread of the warp reads 16 consecutive fp32 columns of its own lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Each thread of the warp writes 16 consecutive fp32 columns of its own lane.
__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float* v) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]),
      "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}

// Each thread of the warp writes 4 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* w) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3])
               : "memory");
}

// Each thread of the warp writes 16 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]),
      "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor, 128-byte swizzle. `lbo`/`sbo` in bytes.
//   K-major operand: rows of 128 B (64 bf16 along K), 8-row swizzle atoms of
//     1024 B stacked along M/N at `sbo`; `lbo` unused.
//   MN-major operand: 64 bf16 along M/N per 128 B row, K rows of 128 B; the
//     next 64 M/N elements sit `lbo` bytes further; 8-row K groups at `sbo`.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, dense, M x N tile.
// a_mn / b_mn = 1 selects an M/N-major (transposed) operand.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                        // D format: fp32
         | (1u << 7)                      // A format: bf16
         | (1u << 10)                     // B format: bf16
         | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);    // M / 16
}

// ------------------------------------------------------------------ misc
// 2^x with the hardware approximation (ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(h);
}

__device__ __forceinline__ void red_add(float* addr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

}  // namespace ptx
}  // namespace aa
