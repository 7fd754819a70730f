// Device layer of the fused linear cross-entropy library for sm_103a:
// inline-PTX wrappers for mbarrier, TMA and the 5th-generation tensor cores
// (tcgen05 + tensor memory), a persistent warp-specialised contraction
// kernel, and the epilogues that fold the loss arithmetic into it.
//
// Contraction D[M,N] = A[M,K] * B[K,N], bf16 operands, fp32 accumulation in
// tensor memory (TMEM). One CTA per SM; 6 warps:
//   warp 0      TMA producer (one lane): streams A/B k-slices into a 4-stage
//               shared-memory ring, 128-byte swizzled;
//   warp 1      MMA issuer (one lane): tcgen05.mma 128x256x16 into one of two
//               256-column TMEM accumulators (double buffered);
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter of the
//               accumulator, then the fused loss arithmetic; bf16 chunk
//               outputs leave through shared-memory boxes and TMA stores.
// A CTA-pair variant (k_gemm_pair, cta_group::2, 256 x 256 tiles, 6-stage
// ring) shares the roles and epilogues. Producers may pace themselves in
// waves of output tiles on a workspace counter (GemmGeom::wave_ctr).
// Every mbarrier wait is bounded in time: on expiry the kernel raises a
// timeout bit in the error word, the other roles see a shared abort flag,
// in-flight copies and MMAs are drained (again bounded) and TMEM is freed.
#pragma once
#include <cuda_bf16.h>
#include <math.h>

#include "lce_internal.h"

namespace lce {

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// shared memory, mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                   bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Context of the bounded waits of one CTA.
struct WaitCtx {
  volatile uint32_t* abort;  // shared flag: some role gave up
  unsigned* err;             // global error word
  uint64_t timeout_ns;
};

// Wait until the phase of `bar` with parity `parity` has completed. Gives up
// after ctx.timeout_ns (sets the abort flag and the timeout bit) or, when
// honor_abort is set, as soon as another role has raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const WaitCtx& ctx,
                                          bool honor_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *ctx.abort) return false;
    if (globaltimer_ns() - t0 > ctx.timeout_ns) {
      *ctx.abort = 1u;
      atomicOr(ctx.err, ERRBIT_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm))
               : "memory");
}

// 2-D tiled load of one box into shared memory; completes on `bar` with the
// box's byte count. c0 is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm,
                                            int32_t c0, int32_t c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// TMA bulk store of one 2D box from this CTA's shared memory to global
// memory (bulk-group completion), and the group bookkeeping around it.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm,
                                             uint32_t src, int32_t c0,
                                             int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], "
      "[%1];" ::"l"(reinterpret_cast<uint64_t>(tm)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most one committed group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Wait until no committed group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed group has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Make this thread's ordinary shared-memory writes visible to TMA reads.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a,
                                             uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 / tensor memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst_smem),
      "r"(ncols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle, tcgen05 version bits.
//   K-major operand (rows of 64 K-elements = 128 B, 8-row atoms of 1 KB):
//     SBO = 1024 (next 8 rows), LBO unused; a K step of 16 adds 32 B.
//   MN-major operand (rows of 64 MN-elements, one row per k, 8-k atoms):
//     SBO = 1024 (next 8 k), LBO = byte distance to the next 64 MN-elements;
//     a K step of 16 adds 16 rows = 2048 B.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo,
                                                uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16) |
         (static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32) |
         (1ull << 46) |  // descriptor version (tcgen05)
         (2ull << 61);   // swizzle: 128 B
}

// Instruction descriptor for kind::f16: bf16 x bf16 -> fp32, M = 128, N = 256.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ constexpr uint32_t idesc_bf16_f32() {
  return (1u << 4) |                                 // D format: f32
         (1u << 7) |                                 // A format: bf16
         (1u << 10) |                                // B format: bf16
         (static_cast<uint32_t>(A_MN) << 15) |       // A major
         (static_cast<uint32_t>(B_MN) << 16) |       // B major
         (static_cast<uint32_t>(BN >> 3) << 17) |    // N / 8
         (static_cast<uint32_t>(BM >> 4) << 24);     // M / 16
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc,
                                       uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape),
// waited on inside the same asm block so no use can move above the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's TMEM lane (32x32b.x64), as
// tmem_ld32: one load for twice the columns, so an epilogue that walks a
// tile waits for half as many loads.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Two fp32 lanes in one 64-bit register pair, for the paired fp32
// instructions (fma/add .rn.f32x2): each lane rounds exactly as the scalar
// instruction does, so a paired loop gives the scalar loop's bits.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
  __nv_bfloat16 v = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&v);
}

__device__ __forceinline__ bool label_valid(int64_t y, int64_t V,
                                            int64_t ignore_index) {
  return y != ignore_index && y >= 0 && y < V;
}

// Column of label y within a contraction over the vocabulary slice
// [v0, v0 + n) of a vocabulary of v_total (v_total 0: the whole vocabulary,
// v_total = n, v0 = 0): -1 when y is not in the slice. *takes_part: y is a
// valid id of the whole vocabulary.
__device__ __forceinline__ int label_column(int64_t y, int64_t n, int64_t v0,
                                            int64_t v_total,
                                            int64_t ignore_index,
                                            bool* takes_part) {
  const int64_t vt = v_total > 0 ? v_total : n;
  *takes_part = label_valid(y, vt, ignore_index);
  const int64_t yl = y - v0;
  return (*takes_part && yl >= 0 && yl < n) ? static_cast<int>(yl) : -1;
}

// ---------------------------------------------------------------------------
// wave pacing (GemmGeom::wave_ctr)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void wave_wait(const GemmGeom& g, uint32_t target) {
  if (!g.wave_ctr || target == 0) return;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];"
                 : "=r"(v)
                 : "l"(g.wave_ctr)
                 : "memory");
    if (v >= target) return;
    if (globaltimer_ns() - t0 > g.wave_wait_ns) return;
    __nanosleep(64);
  }
}

__device__ __forceinline__ void wave_arrive(const GemmGeom& g) {
  if (g.wave_ctr) atomicAdd(g.wave_ctr, 1u);
}

__device__ __forceinline__ void wave_finish(const GemmGeom& g, uint32_t done) {
  if (g.wave_ctr && g.wave_steps > done)
    atomicAdd(g.wave_ctr, g.wave_steps - done);
}

// ---------------------------------------------------------------------------
// unit decode
// ---------------------------------------------------------------------------
struct Unit {
  int m_blk, split, n_first, n_count;
  int64_t row0;  // first output row held in this CTA's accumulator
};

// rows_per_unit = BM for single-CTA tiles, 2 * BM for CTA-pair tiles (the
// pair's second CTA holds rows row0 + BM ...).
__device__ __forceinline__ Unit decode_unit(const GemmGeom& g, int u,
                                            int rows_per_unit = BM,
                                            int rank = 0) {
  Unit t;
  if (g.group_n > 0 && g.tiles_per_split == 1) {
    // groups of group_n column tiles; within a group, row blocks vary
    // slowest so consecutive units share a row panel
    const int per_group = g.num_m * g.group_n;
    const int grp = u / per_group;
    const int r = u - grp * per_group;
    const int n0 = grp * g.group_n;
    const int width = min(g.group_n, g.num_n - n0);
    t.m_blk = r / width;
    t.split = n0 + (r - t.m_blk * width);
    t.n_first = t.split;
    t.n_count = 1;
  } else {
    t.m_blk = u / g.splits;
    t.split = u - t.m_blk * g.splits;
    t.n_first = t.split * g.tiles_per_split;
    t.n_count = min(g.tiles_per_split, g.num_n - t.n_first);
  }
  t.row0 = static_cast<int64_t>(t.m_blk) * rows_per_unit +
           static_cast<int64_t>(rank) * BM;
  return t;
}

// ---------------------------------------------------------------------------
// epilogues: one thread per accumulator row, 32 columns per TMEM load
// ---------------------------------------------------------------------------

// Over the first nv (1..64) of one 64-column TMEM load, four interleaved
// partials each: the largest value, and the sum (label smoothing's logit
// sums). A whole piece (nv == 64, warp-uniform) runs without column guards.
__device__ __forceinline__ float piece_max(const float (&v)[64], int nv) {
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if (nv == 64) {
#pragma unroll
    for (int i = 0; i < 64; i += 8) {
      mx[0] = max3(mx[0], v[i], v[i + 1]);
      mx[1] = max3(mx[1], v[i + 2], v[i + 3]);
      mx[2] = max3(mx[2], v[i + 4], v[i + 5]);
      mx[3] = max3(mx[3], v[i + 6], v[i + 7]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i < nv) mx[i & 3] = fmaxf(mx[i & 3], v[i]);
  }
  return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}
__device__ __forceinline__ float piece_sum(const float (&v)[64], int nv) {
  float za[4] = {0.f, 0.f, 0.f, 0.f};
  if (nv == 64) {
#pragma unroll
    for (int i = 0; i < 64; ++i) za[i & 3] += v[i];
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i)
      if (i < nv) za[i & 3] += v[i];
  }
  return (za[0] + za[1]) + (za[2] + za[3]);
}

// What every epilogue may use besides its parameters: the store map and
// the two shared-memory staging buffers of this warp (EPI_BUF_BYTES each,
// 1 KB aligned, for 64-byte-swizzled EPI_BOX x EPI_BOX bf16 boxes), and how
// many boxes this warp has handed to TMA so far. Set by the epilogue role.
struct EpiBase {
  const CUtensorMap* te = nullptr;
  uint32_t stage = 0;
  uint32_t nstored = 0;

  // Warp-collective: the 32 x 32 bf16 box of this warp's rows [wrow0,
  // wrow0 + 32) and columns [j0, j0 + 32), lane l holding row wrow0 + l in
  // v, goes through this warp's next staging buffer (row r at r * 64 bytes,
  // its 16-byte pieces in 64-byte-swizzle order) and out by one TMA store,
  // which drops the rows and columns past the map's extent. Two buffers
  // alternate; a buffer is reused once the store before last has read it.
  __device__ __forceinline__ void store_box(const float (&v)[32], int64_t j0,
                                            int64_t wrow0,
                                            const CUtensorMap* map = nullptr) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    store_box_words(w, j0, wrow0, map);
  }

  // The same box from bf16 pairs already packed (w[i] = columns 2i, 2i + 1
  // of this lane's row), through `map` (NULL: te).
  __device__ __forceinline__ void store_box_words(const uint32_t (&w)[16],
                                                  int64_t j0, int64_t wrow0,
                                                  const CUtensorMap* map) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t buf = stage + (nstored & 1u) * EPI_BUF_BYTES;
    if (lane == 0 && nstored >= 2) bulk_wait_read1();
    __syncwarp();
    const uint32_t rowa = buf + lane * 64u;
    const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_shared_v4(rowa + ((static_cast<uint32_t>(q) ^ sw) << 4), w[4 * q],
                   w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map ? map : te, buf, static_cast<int32_t>(j0),
                   static_cast<int32_t>(wrow0));
      bulk_commit();
    }
    ++nstored;
  }

  // Both 32-column boxes of a 64-column piece at once, columns [j0, j0 +
  // 32) from w0 and, when `second`, [j0 + 32, j0 + 64) from w1: the two
  // buffers filled together, one proxy fence, both stores in one group
  // (half the fences and warp syncs of two store_box_words calls). An
  // epilogue uses either this or store_box_words, never both, since this
  // takes both buffers at once.
  __device__ __forceinline__ void store_box_pair(const uint32_t (&w0)[16],
                                                 const uint32_t (&w1)[16],
                                                 int64_t j0, int64_t wrow0,
                                                 bool second) {
    const uint32_t lane = threadIdx.x & 31u;
    if (lane == 0 && nstored > 0) bulk_wait_read0();
    __syncwarp();
    const uint32_t rowa = stage + lane * 64u;
    const uint32_t rowb = rowa + EPI_BUF_BYTES;
    const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_shared_v4(rowa + ((static_cast<uint32_t>(q) ^ sw) << 4), w0[4 * q],
                   w0[4 * q + 1], w0[4 * q + 2], w0[4 * q + 3]);
    if (second) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_shared_v4(rowb + ((static_cast<uint32_t>(q) ^ sw) << 4), w1[4 * q],
                     w1[4 * q + 1], w1[4 * q + 2], w1[4 * q + 3]);
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(te, stage, static_cast<int32_t>(j0),
                   static_cast<int32_t>(wrow0));
      if (second)
        tma_store_2d(te, stage + EPI_BUF_BYTES, static_cast<int32_t>(j0 + 32),
                     static_cast<int32_t>(wrow0));
      bulk_commit();
    }
    ++nstored;
  }
};

// Forward: per-row running (max, sum 2^(u-max)) in log2 units over the
// unit's columns; the logit at the label is written by the one tile that
// holds that column.
struct EpiLse : EpiBase {
  using Params = LseParams;
  float m2, s;
  float zs;  // sum of the unit's logits (label smoothing only)
  int64_t row;
  int yv;  // label if it takes part, else -1
  bool row_ok;

  __device__ __forceinline__ void begin_unit(const Params& p, const GemmGeom& g,
                                             const Unit& t, int r) {
    row = t.row0 + r;
    row_ok = row < g.M;
    yv = -1;
    if (row_ok) {
      bool takes;
      yv = label_column(p.labels[row], g.N, p.v0, p.v_total, p.ignore_index,
                        &takes);
    }
    m2 = -INFINITY;
    s = 0.f;
    zs = 0.f;
  }

  __device__ __forceinline__ void tile(const Params& p, const GemmGeom& g,
                                       const Unit&, int n_blk, uint32_t taddr,
                                       int) {
    const int64_t n0 = static_cast<int64_t>(n_blk) * BN;
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      const int64_t j0 = n0 + c * 64;
      if (j0 >= g.N) break;  // same for the whole warp
      float v[64];
      tmem_ld64(taddr + c * 64, v);
      const int64_t rem = g.N - j0;
      const int nv = rem < 64 ? static_cast<int>(rem) : 64;
      const int yo = yv - static_cast<int>(j0);
      if (static_cast<unsigned>(yo) < 64u) {
        float zyv = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i == yo) zyv = v[i];
        p.zy[row] = zyv;
      }
      if (p.part_z != nullptr) zs += piece_sum(v, nv);  // warp-uniform
      // max(v) log2 e is max(v log2 e) exactly (rounding is monotone)
      const float mn = fmaxf(m2, piece_max(v, nv) * LOG2E);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (nv == 64) {  // warp-uniform: a whole piece, no column guards
        const uint64_t c2 = f2pack(LOG2E, LOG2E), m2n = f2pack(-mn, -mn);
        uint64_t a01 = f2pack(0.f, 0.f), a23 = a01;  // acc[0..1], acc[2..3]
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          float x0, x1;
          f2unpack(fma2(f2pack(v[i], v[i + 1]), c2, m2n), x0, x1);
          const uint64_t e = f2pack(ex2(x0), ex2(x1));
          if ((i & 2) == 0)
            a01 = add2(a01, e);
          else
            a23 = add2(a23, e);
        }
        f2unpack(a01, acc[0], acc[1]);
        f2unpack(a23, acc[2], acc[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i < nv) acc[i & 3] += ex2(fmaf(v[i], LOG2E, -mn));
      }
      s = s * ex2(m2 - mn) + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
      m2 = mn;
    }
  }

  __device__ __forceinline__ void end_unit(const Params& p, const GemmGeom& g,
                                           const Unit& t, int) {
    if (row_ok) {
      p.part_m[static_cast<int64_t>(t.split) * g.M + row] = m2;
      p.part_s[static_cast<int64_t>(t.split) * g.M + row] = s;
      if (p.part_z != nullptr)
        p.part_z[static_cast<int64_t>(t.split) * g.M + row] = zs;
    }
  }
};

// Backward recompute: G = exp(z - lse) - [j == y] for rows that take part,
// 0 for the others, rounded to bf16 and written by TMA stores of staged
// 32 x 32 boxes (EpiBase::store_box). With a loss variant, G = zf exp(z -
// lse) - ome [j == y] - eps_v (VariantGrad); the plain constants {1, 1, 0}
// leave every value's bits as the plain formula gives them. The dloss/N
// scale is applied later, in fp32, by the dH and dW epilogues.
struct EpiGrad : EpiBase {
  using Params = GradParams;
  int64_t row;
  bool row_ok;
  bool takes;  // the row takes part in the loss
  int yv;      // label column in this contraction, or -1
  float lse2;  // lse log2 e; +inf for a row that does not take part
  float zf;    // 1 + 2 zcoef lse (1 for the plain loss); 0 if not taking part
  float epsr;  // eps_v, or 0 for a row that does not take part

  __device__ __forceinline__ void begin_unit(const Params& p, const GemmGeom& g,
                                             const Unit& t, int r) {
    row = t.row0 + r;
    row_ok = row < g.M;
    takes = false;
    yv = -1;
    if (row_ok)
      yv = label_column(p.labels[row], g.N, p.v0, p.v_total, p.ignore_index,
                        &takes);
    // a row that does not take part gets 2^-inf * 0 - 0 = +0 everywhere
    // from the same formula as the others, without a select per element
    lse2 = INFINITY;
    zf = 0.f;
    epsr = 0.f;
    if (takes) {
      lse2 = p.lse[row] * LOG2E;
      zf = fmaf(p.var.zloss2, p.lse[row], 1.f);
      epsr = p.var.eps_v;
    }
  }

  __device__ __forceinline__ void tile(const Params& p, const GemmGeom& g,
                                       const Unit&, int n_blk, uint32_t taddr,
                                       int) {
    const int64_t n0 = static_cast<int64_t>(n_blk) * BN;
    // rows past M and columns past N hold junk that the store drops
    const int64_t wrow0 = row - static_cast<int64_t>(threadIdx.x & 31);
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      const int64_t j0 = n0 + c * 64;
      if (j0 >= g.N) break;
      float v[64];
      tmem_ld64(taddr + c * 64, v);
      const int yo = yv - static_cast<int>(j0);
      uint32_t w0[16], w1[16];
      if (static_cast<unsigned>(yo) >= 64u) {
        // no label in this piece (all but ~64 / V of the rows' pieces; the
        // branch is per row, so a warp rarely takes both sides)
        const uint64_t c2 = f2pack(LOG2E, LOG2E), l2 = f2pack(-lse2, -lse2);
        const uint64_t z2 = f2pack(zf, zf), e2 = f2pack(-epsr, -epsr);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          float x0, x1, g0, g1;
          f2unpack(fma2(f2pack(v[i], v[i + 1]), c2, l2), x0, x1);
          f2unpack(fma2(f2pack(ex2(x0), ex2(x1)), z2, e2), g0, g1);
          if (i < 32)
            w0[i / 2] = pack_bf16x2(g0, g1);
          else
            w1[(i - 32) / 2] = pack_bf16x2(g0, g1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          float gi[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            gi[k] = fmaf(ex2(fmaf(v[i + k], LOG2E, -lse2)), zf, -epsr);
            if (i + k == yo) gi[k] -= p.var.ome;
          }
          if (i < 32)
            w0[i / 2] = pack_bf16x2(gi[0], gi[1]);
          else
            w1[(i - 32) / 2] = pack_bf16x2(gi[0], gi[1]);
        }
      }
      if (wrow0 < g.M)  // warp-uniform test
        store_box_pair(w0, w1, j0, wrow0, j0 + 32 < g.N);
    }
  }

  __device__ __forceinline__ void end_unit(const Params&, const GemmGeom&,
                                           const Unit&, int) {}
};

// Fused forward+backward over one row chunk. Two passes over each tile's
// TMEM columns: the first finds the tile's row maximum m_t (log2 units) and
// gathers the label logit; the second writes e = 2^(u - m_t) in bf16
// (staged 32 x 32 boxes, TMA stores) and sums the fp32 values. (m_t, sum) then merge into the row's running
// (max, sum) exactly as in EpiLse, and m_t is stored so that a later pass
// can turn e into softmax - onehot once the row's lse is known.
struct EpiFused : EpiBase {
  using Params = FusedParams;
  float m2, s;
  float zs;  // sum of the unit's logits (label smoothing only)
  int64_t row;
  int yv;
  bool row_ok;

  __device__ __forceinline__ void begin_unit(const Params& p, const GemmGeom& g,
                                             const Unit& t, int r) {
    row = t.row0 + r;
    row_ok = row < g.M;
    yv = -1;
    if (row_ok) {
      bool takes;
      yv = label_column(p.labels[row], g.N, p.v0, p.v_total, p.ignore_index,
                        &takes);
    }
    m2 = -INFINITY;
    s = 0.f;
    zs = 0.f;
  }

  __device__ __forceinline__ void tile(const Params& p, const GemmGeom& g,
                                       const Unit&, int n_blk, uint32_t taddr,
                                       int) {
    const int64_t n0 = static_cast<int64_t>(n_blk) * BN;
    // pass 1: tile maximum, label logit (64 columns per TMEM load)
    float mx = -INFINITY;
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      const int64_t j0 = n0 + c * 64;
      if (j0 >= g.N) break;
      float v[64];
      tmem_ld64(taddr + c * 64, v);
      const int64_t rem = g.N - j0;
      const int nv = rem < 64 ? static_cast<int>(rem) : 64;
      const int yo = yv - static_cast<int>(j0);
      if (static_cast<unsigned>(yo) < 64u) {
        float zyv = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i == yo) zyv = v[i];
        if (row_ok) p.zy[row] = zyv;
      }
      if (p.part_z != nullptr) zs += piece_sum(v, nv);  // warp-uniform
      mx = fmaxf(mx, piece_max(v, nv));
    }
    // max(v) log2 e is max(v log2 e) exactly (rounding is monotone)
    const float mt = mx * LOG2E;
    // pass 2: exponentials relative to the tile maximum. The two 32-column
    // halves of a 64-column load, for the warp's 32 rows, go through two
    // shared-memory boxes (row r at r * 64 bytes, its 16-byte pieces in
    // 64-byte-swizzle order) and out by two TMA stores, which write whole
    // rows' segments and drop the rows past M and the columns past N.
    // the running sums acc[0..3] in two register pairs: a01 = (acc[0],
    // acc[1]), a23 = (acc[2], acc[3]); column i adds into acc[i & 3]
    uint64_t a01 = f2pack(0.f, 0.f), a23 = a01;
    const uint64_t c2 = f2pack(LOG2E, LOG2E), m2n = f2pack(-mt, -mt);
    const int64_t wrow0 = row - static_cast<int64_t>(threadIdx.x & 31);
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      const int64_t j0 = n0 + c * 64;
      if (j0 >= g.N) break;
      float v[64];
      tmem_ld64(taddr + c * 64, v);
      const int64_t rem = g.N - j0;
      const int nv = rem < 64 ? static_cast<int>(rem) : 64;
      uint32_t w0[16], w1[16];
      if (nv == 64) {  // warp-uniform: a whole piece, no column guards
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          float x0, x1;
          f2unpack(fma2(f2pack(v[i], v[i + 1]), c2, m2n), x0, x1);
          const float e0 = ex2(x0), e1 = ex2(x1);
          if ((i & 2) == 0)
            a01 = add2(a01, f2pack(e0, e1));
          else
            a23 = add2(a23, f2pack(e0, e1));
          if (i < 32)
            w0[i / 2] = pack_bf16x2(e0, e1);
          else
            w1[(i - 32) / 2] = pack_bf16x2(e0, e1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float e0 = (i < nv) ? ex2(fmaf(v[i], LOG2E, -mt)) : 0.f;
          const float e1 =
              (i + 1 < nv) ? ex2(fmaf(v[i + 1], LOG2E, -mt)) : 0.f;
          if ((i & 2) == 0)
            a01 = add2(a01, f2pack(e0, e1));
          else
            a23 = add2(a23, f2pack(e0, e1));
          if (i < 32)
            w0[i / 2] = pack_bf16x2(e0, e1);
          else
            w1[(i - 32) / 2] = pack_bf16x2(e0, e1);
        }
      }
      if (wrow0 < g.M)  // warp-uniform test
        store_box_pair(w0, w1, j0, wrow0, j0 + 32 < g.N);
    }
    float acc[4];
    f2unpack(a01, acc[0], acc[1]);
    f2unpack(a23, acc[2], acc[3]);
    const float st = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    const float mn = fmaxf(m2, mt);
    s = s * ex2(m2 - mn) + st * ex2(mt - mn);
    m2 = mn;
    if (row_ok) p.tile_max[row * g.num_n + n_blk] = mt;
  }

  __device__ __forceinline__ void end_unit(const Params& p, const GemmGeom& g,
                                           const Unit& t, int) {
    if (row_ok) {
      p.part_m[static_cast<int64_t>(t.split) * g.M + row] = m2;
      p.part_s[static_cast<int64_t>(t.split) * g.M + row] = s;
      if (p.part_z != nullptr)
        p.part_z[static_cast<int64_t>(t.split) * g.M + row] = zs;
    }
  }
};

// out[row][col] (+)= scale * acc, fp32 or bf16. scale = dloss / N when the
// parameters carry them (N = 0 gives 0; a missing dloss counts as 1), else 1.
struct EpiStore : EpiBase {
  using Params = StoreParams;
  int64_t row;
  bool row_ok;
  float scale;
  void* base;     // output holding this row
  int64_t orow;   // the row's index in it

  __device__ __forceinline__ void begin_unit(const Params& p, const GemmGeom& g,
                                             const Unit& t, int r) {
    row = t.row0 + r;
    row_ok = row < g.M;
    base = p.out;
    orow = row;
    if (p.out2 != nullptr && row >= p.split_row) {
      base = p.out2;
      orow = row - p.split_row;
    }
    scale = 1.f;
    if (p.n_valid != nullptr) {
      const unsigned long long n = *p.n_valid;
      const double d = p.dloss != nullptr ? *p.dloss : 1.0;
      scale = n ? static_cast<float>(d / static_cast<double>(n)) : 0.f;
    } else if (p.dloss != nullptr) {
      scale = *p.dloss;
    }
  }

  __device__ __forceinline__ void tile(const Params& p, const GemmGeom& g,
                                       const Unit&, int n_blk, uint32_t taddr,
                                       int) {
    const int64_t n0 = static_cast<int64_t>(n_blk) * BN;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int64_t j0 = n0 + c * 32;
      if (j0 >= g.N) break;
      float v[32];
      tmem_ld32(taddr + c * 32, v);
      if (!row_ok) continue;
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= scale;
      const bool full = j0 + 32 <= g.N;
      const int nv = full ? 32 : static_cast<int>(g.N - j0);
      if (p.out_f32) {
        float* dst = static_cast<float*>(base) + orow * p.ldo + j0;
        if (full) {
          float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 o = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2],
                                   v[4 * q + 3]);
            if (p.accumulate) {
              const float4 a = d4[q];
              o.x += a.x;
              o.y += a.y;
              o.z += a.z;
              o.w += a.w;
            }
            d4[q] = o;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < nv) dst[i] = p.accumulate ? dst[i] + v[i] : v[i];
        }
      } else {
        uint16_t* dst = static_cast<uint16_t*>(base) + orow * p.ldo + j0;
        if (full) {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]),
                               pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                               pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < nv) dst[i] = to_bf16_bits(v[i]);
        }
      }
    }
  }

  __device__ __forceinline__ void end_unit(const Params&, const GemmGeom&,
                                           const Unit&, int) {}
};

// 1 / (1 + 2^(-t log2 e)): the logistic function on the SFU.
__device__ __forceinline__ float sigmoid_fast(float t) {
  return __fdividef(1.f, 1.f + ex2(-t * LOG2E));
}

// Gated-MLP gate/up contraction with B dual along N: for the tile's 128
// output columns, accumulator columns 0..127 are g and 128..255 are u;
// writes a = silu(g) u (and g, u when asked) in bf16, each 32-column chunk
// of the warp's 32 rows through a staged box and one TMA store (the store
// maps drop the rows past M).
struct EpiSwiGLU : EpiBase {
  using Params = SwigluParams;
  int64_t row;

  __device__ __forceinline__ void begin_unit(const Params&, const GemmGeom&,
                                             const Unit& t, int r) {
    row = t.row0 + r;
  }

  __device__ __forceinline__ void tile(const Params& p, const GemmGeom& g,
                                       const Unit&, int n_blk, uint32_t taddr,
                                       int) {
    const int64_t i0 = static_cast<int64_t>(n_blk) * (BN / 2);
    const int64_t wrow0 = row - static_cast<int64_t>(threadIdx.x & 31);
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      const int64_t j0 = i0 + c * 32;
      if (j0 >= g.N) break;
      float gv[32], uv[32];
      tmem_ld32(taddr + c * 32, gv);
      tmem_ld32(taddr + BN / 2 + c * 32, uv);
      if (wrow0 >= g.M) continue;  // warp-uniform: all of the warp's rows
      if (p.save_gu) {
        store_box(gv, j0, wrow0, &p.map_g);
        store_box(uv, j0, wrow0, &p.map_u);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) uv[i] *= gv[i] * sigmoid_fast(gv[i]);
      store_box(uv, j0, wrow0, &p.map_a);
    }
  }

  __device__ __forceinline__ void end_unit(const Params&, const GemmGeom&,
                                           const Unit&, int) {}
};

// Gated-MLP backward: accumulator = da; dg = da u silu'(g),
// du = da silu(g), with silu'(t) = s (1 + t (1 - s)), s the logistic.
// I is a multiple of 64 (checked by the host), so every 32-column chunk is
// whole; g and u of a chunk are loaded one chunk ahead (per thread, its own
// row), dg and du leave through staged boxes and TMA stores of [dg | du].
struct EpiSwiGLUBwd : EpiBase {
  using Params = SwigluBwdParams;
  int64_t row;
  bool row_ok;

  __device__ __forceinline__ void begin_unit(const Params&, const GemmGeom& g,
                                             const Unit& t, int r) {
    row = t.row0 + r;
    row_ok = row < g.M;
  }

  // g and u of one 32-column chunk: 4 x 16-byte vectors each
  struct GU {
    uint4 g[4], u[4];
  };

  __device__ __forceinline__ void load_gu(const Params& p, int64_t j0,
                                          GU& b) const {
    const uint4* gp = reinterpret_cast<const uint4*>(p.g + row * p.ld_gu + j0);
    const uint4* up = reinterpret_cast<const uint4*>(p.u + row * p.ld_gu + j0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      b.g[q] = gp[q];
      b.u[q] = up[q];
    }
  }

  __device__ __forceinline__ void tile(const Params& p, const GemmGeom& g,
                                       const Unit&, int n_blk, uint32_t taddr,
                                       int) {
    const int64_t n0 = static_cast<int64_t>(n_blk) * BN;
    const int64_t wrow0 = row - static_cast<int64_t>(threadIdx.x & 31);
    GU nxt;
    if (row_ok && n0 < g.N) load_gu(p, n0, nxt);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int64_t j0 = n0 + c * 32;
      if (j0 >= g.N) break;
      const GU cur = nxt;
      if (row_ok && c + 1 < BN / 32 && j0 + 32 < g.N) load_gu(p, j0 + 32, nxt);
      float da[32];
      tmem_ld32(taddr + c * 32, da);
      if (wrow0 >= g.M) continue;  // warp-uniform: all of the warp's rows
      // rows past M compute from unloaded g, u; their boxes' rows are
      // dropped by the store map
      uint32_t og[16], ou[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t gw[4] = {cur.g[q].x, cur.g[q].y, cur.g[q].z, cur.g[q].w};
        const uint32_t uw[4] = {cur.u[q].x, cur.u[q].y, cur.u[q].z, cur.u[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float dgv[2], duv[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float gx = __uint_as_float(h ? (gw[e] & 0xFFFF0000u)
                                               : (gw[e] << 16));
            const float ux = __uint_as_float(h ? (uw[e] & 0xFFFF0000u)
                                               : (uw[e] << 16));
            const float sg = sigmoid_fast(gx);
            const float d = da[8 * q + 2 * e + h];
            duv[h] = d * gx * sg;
            dgv[h] = d * ux * sg * (1.f + gx * (1.f - sg));
          }
          og[4 * q + e] = pack_bf16x2(dgv[0], dgv[1]);
          ou[4 * q + e] = pack_bf16x2(duv[0], duv[1]);
        }
      }
      store_box_words(og, j0, wrow0, &p.map_dgu);
      store_box_words(ou, p.du_off + j0, wrow0, &p.map_dgu);
    }
  }

  __device__ __forceinline__ void end_unit(const Params&, const GemmGeom&,
                                           const Unit&, int) {}
};

// ---------------------------------------------------------------------------
// the persistent contraction kernel
// ---------------------------------------------------------------------------
struct SmemMap {
  uint32_t a, b, bars;
  __device__ __forceinline__ uint32_t full(int s) const { return bars + 8u * s; }
  __device__ __forceinline__ uint32_t empty(int s) const {
    return bars + 8u * (STAGES + s);
  }
  __device__ __forceinline__ uint32_t tfull(int a_) const {
    return bars + 8u * (2 * STAGES + a_);
  }
  __device__ __forceinline__ uint32_t tempty(int a_) const {
    return bars + 8u * (2 * STAGES + 2 + a_);
  }
  __device__ __forceinline__ uint32_t drain() const {
    return bars + 8u * (2 * STAGES + 4);
  }
};

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void role_producer(const CUtensorMap* ta,
                                              const CUtensorMap* tb,
                                              const CUtensorMap* tb2,
                                              const GemmGeom& g,
                                              const SmemMap& sm,
                                              const WaitCtx& ctx) {
  uint32_t stage = 0, phase = 0, issued = 0;
  bool ok = true;
  uint32_t step = 0;  // output tiles whose loads this CTA has issued
  for (int u = blockIdx.x; ok && u < g.num_units; u += gridDim.x) {
    const Unit t = decode_unit(g, u);
    const int m0 = t.m_blk * BM;
    for (int tt = 0; ok && tt < t.n_count; ++tt) {
      wave_wait(g, step * gridDim.x);
      const int n0 = (t.n_first + tt) * BN;
      for (int kb = 0; kb < g.num_kb; ++kb) {
        if (!mbar_wait(sm.empty(stage), phase ^ 1u, ctx, true)) {
          ok = false;
          break;
        }
        const uint32_t fb = sm.full(stage);
        mbar_arrive_expect_tx(fb, STAGE_BYTES);
        const uint32_t sa = sm.a + stage * A_STAGE_BYTES;
        const uint32_t sb = sm.b + stage * B_STAGE_BYTES;
        const int k0 = kb * BK;
        if (A_MN) {
#pragma unroll
          for (int j = 0; j < BM / 64; ++j)
            tma_load_2d(sa + j * 64 * BK * 2, ta, m0 + 64 * j, k0, fb);
        } else {
          tma_load_2d(sa, ta, k0, m0, fb);
        }
        // B from the second map past the K split (dual along K)
        const bool second = g.b_dual == 2 && kb >= g.k_split_kb;
        const CUtensorMap* tbk = second ? tb2 : tb;
        const int kq = second ? k0 - g.k_split_kb * BK : k0;
        if (B_MN) {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(sb + j * 64 * BK * 2, tbk, n0 + 64 * j, kq, fb);
        } else if (g.b_dual == 1) {
          // dual along N: 128 rows of each map, same rows
          const int nr = (t.n_first + tt) * (BN / 2);
          tma_load_2d(sb, tb, k0, nr, fb);
          tma_load_2d(sb + (BN / 2) * BK * 2, tb2, k0, nr, fb);
        } else {
          tma_load_2d(sb, tbk, kq, n0, fb);
        }
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        wave_arrive(g);
        ++step;
      }
    }
  }
  wave_finish(g, step);
  // Drain: every copy issued must have landed before the CTA may exit.
  for (int s = 0; s < STAGES; ++s) {
    const uint32_t cnt = issued / STAGES + (static_cast<uint32_t>(s) < issued % STAGES ? 1u : 0u);
    if (cnt) mbar_wait(sm.full(s), (cnt - 1u) & 1u, ctx, false);
  }
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void role_mma(const GemmGeom& g, const SmemMap& sm,
                                         uint32_t tmem_base,
                                         const WaitCtx& ctx) {
  constexpr uint32_t IDESC = idesc_bf16_f32<A_MN, B_MN>();
  // operand strides inside one stage (see sdesc_sw128)
  constexpr uint32_t MN_LBO = 64 * BK * 2;  // one 64-wide MN box: 8 KB
  uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < g.num_units; u += gridDim.x) {
    const Unit t = decode_unit(g, u);
    for (int tt = 0; ok && tt < t.n_count; ++tt) {
      if (!mbar_wait(sm.tempty(acc), acc_phase ^ 1u, ctx, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + acc * BN;
      for (int kb = 0; kb < g.num_kb; ++kb) {
        if (!mbar_wait(sm.full(stage), phase, ctx, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = sm.a + stage * A_STAGE_BYTES;
        const uint32_t sb = sm.b + stage * B_STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t ad = A_MN ? sdesc_sw128(sa + k * 2048, MN_LBO, 1024)
                                   : sdesc_sw128(sa + k * 32, 16, 1024);
          const uint64_t bd = B_MN ? sdesc_sw128(sb + k * 2048, MN_LBO, 1024)
                                   : sdesc_sw128(sb + k * 32, 16, 1024);
          tc_mma(d, ad, bd, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(sm.empty(stage));  // frees the stage once these MMAs finish
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(sm.tfull(acc));  // accumulator ready for the epilogue
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  // Drain: all MMAs issued by this thread complete before TMEM is freed.
  tc_commit(sm.drain());
  mbar_wait(sm.drain(), 0, ctx, false);
}

template <class Epi>
__device__ __forceinline__ void role_epilogue(const GemmGeom& g,
                                              const typename Epi::Params& p,
                                              const SmemMap& sm,
                                              uint32_t tmem_base,
                                              const WaitCtx& ctx, int warp,
                                              int lane, const CUtensorMap* te,
                                              uint32_t stage_base) {
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  const int r = q * 32 + lane;
  uint32_t acc = 0, acc_phase = 0;
  Epi epi;
  epi.te = te;
  epi.stage = stage_base + static_cast<uint32_t>(q) * 2u * EPI_BUF_BYTES;
  for (int u = blockIdx.x; u < g.num_units; u += gridDim.x) {
    const Unit t = decode_unit(g, u);
    epi.begin_unit(p, g, t, r);
    bool ok = true;
    for (int tt = 0; tt < t.n_count; ++tt) {
      const bool got = mbar_wait(sm.tfull(acc), acc_phase, ctx, true);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      epi.tile(p, g, t, t.n_first + tt, taddr, r);
      tc_fence_before();
      mbar_arrive(sm.tempty(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) break;
    epi.end_unit(p, g, t, r);
  }
  // every TMA store of this warp has finished reading shared memory and
  // writing global memory before the CTA may exit
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

template <class Epi, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap ta,
           const __grid_constant__ CUtensorMap tb,
           const __grid_constant__ CUtensorMap tb2, const GemmGeom g,
           const __grid_constant__ typename Epi::Params p, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms: 1 KB aligned
  SmemMap sm;
  sm.a = base;
  sm.b = base + STAGES * A_STAGE_BYTES;
  sm.bars = base + STAGES * STAGE_BYTES;
  uint8_t* misc = smem_raw + (sm.bars - raw) + 8 * (2 * STAGES + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(sm.full(s), 1);
      mbar_init(sm.empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(sm.tfull(a), 1);
      mbar_init(sm.tempty(a), 128);  // every epilogue thread arrives
    }
    mbar_init(sm.drain(), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&ta);
    tma_prefetch_desc(&tb);
    if (g.b_dual) tma_prefetch_desc(&tb2);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx ctx{abort_flag, err, g.timeout_ns};

  if (warp == 0) {
    if (lane == 0) role_producer<A_MN, B_MN>(&ta, &tb, &tb2, g, sm, ctx);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) role_mma<A_MN, B_MN>(g, sm, tmem_base, ctx);
    __syncwarp();
  } else {
    role_epilogue<Epi>(g, p, sm, tmem_base, ctx, warp, lane, &tb2,
                       base + STAGES * STAGE_BYTES + 1024);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Host helper for the kernel translation units: launch one instantiation.
template <class Epi, bool A_MN, bool B_MN>
cudaError_t launch_gemm_t(const CUtensorMap& ta, const CUtensorMap& tb,
                          const GemmGeom& g, const typename Epi::Params& p,
                          unsigned* err, int grid, cudaStream_t s,
                          const CUtensorMap* tb2 = nullptr) {
  auto kern = k_gemm<Epi, A_MN, B_MN>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, GEMM_THREADS, GEMM_SMEM_BYTES, s>>>(ta, tb, tb2 ? *tb2 : tb, g,
                                                   p, err);
  return cudaGetLastError();
}

// ===========================================================================
// CTA-pair contraction (tcgen05 cta_group::2): a cluster of two CTAs on two
// SMs computes one 256 x 256 output tile. Each CTA loads 128 rows of A and
// 128 rows (columns of the output) of B per k-slice into its own shared
// memory; the pair's first CTA (the leader) issues 256x256x16 MMAs that read
// both CTAs' operands and write rows 0..127 into its own TMEM and rows
// 128..255 into its peer's. Per CTA a stage is 32 KB instead of 48 KB, so the
// ring is 6 deep, and the B operand is read from shared memory once per pair.
//   - full[s]    (leader's): the leader's producer posts the stage's bytes of
//                both CTAs; both CTAs' TMA copies complete on it;
//   - empty[s]   (each CTA's): the leader's commit arrives on both;
//   - tfull[a]   (each CTA's): the leader's commit arrives on both;
//   - tempty[a]  (leader's): one arrival per epilogue warp of both CTAs.
// ===========================================================================
constexpr int STAGES2 = 6;
constexpr int A2_STAGE_BYTES = BM * BK * 2;  // 16 KB
constexpr int B2_STAGE_BYTES = BM * BK * 2;  // 16 KB: half of the 256 columns
constexpr int STAGE2_BYTES = A2_STAGE_BYTES + B2_STAGE_BYTES;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (either CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile(
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
          cluster_addr)
      : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion is counted
// on an mbarrier of either CTA of the pair (given as a cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst,
                                                 const CUtensorMap* tm,
                                                 int32_t c0, int32_t c1,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile."
      "mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1),
      "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem,
                                                uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst_smem),
      "r"(ncols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr,
                                                  uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc,
                                            uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this shared offset in both CTAs of the pair once
// this thread's tcgen05 operations have completed.
__device__ __forceinline__ void tc_commit_pair_both(uint32_t bar) {
  const uint16_t mask = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster."
      "multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ constexpr uint32_t idesc_pair_bf16_f32() {
  return (1u << 4) | (1u << 7) | (1u << 10) |
         (static_cast<uint32_t>(A_MN) << 15) |
         (static_cast<uint32_t>(B_MN) << 16) |
         (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>((2 * BM) >> 4) << 24);  // M = 256
}

struct SmemMap2 {
  uint32_t a, b, bars;
  __device__ __forceinline__ uint32_t full(int s) const { return bars + 8u * s; }
  __device__ __forceinline__ uint32_t empty(int s) const {
    return bars + 8u * (STAGES2 + s);
  }
  __device__ __forceinline__ uint32_t tfull(int a_) const {
    return bars + 8u * (2 * STAGES2 + a_);
  }
  __device__ __forceinline__ uint32_t tempty(int a_) const {
    return bars + 8u * (2 * STAGES2 + 2 + a_);
  }
  __device__ __forceinline__ uint32_t drain() const {
    return bars + 8u * (2 * STAGES2 + 4);
  }
};

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void role_producer_pair(const CUtensorMap* ta,
                                                   const CUtensorMap* tb,
                                                   const CUtensorMap* tb2,
                                                   const GemmGeom& g,
                                                   const SmemMap2& sm,
                                                   uint32_t rank,
                                                   const WaitCtx& ctx) {
  const bool leader = rank == 0;
  const int nclusters = gridDim.x >> 1;
  const int cluster = blockIdx.x >> 1;
  uint32_t stage = 0, phase = 0, issued = 0;
  bool ok = true;
  uint32_t step = 0;  // output tiles whose loads this CTA has issued
  for (int u = cluster; ok && u < g.num_units; u += nclusters) {
    const Unit t = decode_unit(g, u, 2 * BM, static_cast<int>(rank));
    const int a0 = static_cast<int>(t.row0);  // this CTA's 128 rows of A
    for (int tt = 0; ok && tt < t.n_count; ++tt) {
      if (leader) wave_wait(g, step * static_cast<uint32_t>(nclusters));
      // this CTA's 128 of the tile's 256 output columns; dual along N: the
      // leader takes the first map's 128 rows, the peer the second's
      const bool dual_n = g.b_dual == 1;
      const int b0 = dual_n ? (t.n_first + tt) * BM
                            : (t.n_first + tt) * BN + static_cast<int>(rank) * BM;
      const CUtensorMap* tbn = (dual_n && rank == 1) ? tb2 : tb;
      for (int kb = 0; kb < g.num_kb; ++kb) {
        if (!mbar_wait(sm.empty(stage), phase ^ 1u, ctx, true)) {
          ok = false;
          break;
        }
        const uint32_t fb = mapa_shared(sm.full(stage), 0);
        if (leader) mbar_arrive_expect_tx(sm.full(stage), 2 * STAGE2_BYTES);
        const uint32_t sa = sm.a + stage * A2_STAGE_BYTES;
        const uint32_t sb = sm.b + stage * B2_STAGE_BYTES;
        const int k0 = kb * BK;
        if (A_MN) {
#pragma unroll
          for (int j = 0; j < BM / 64; ++j)
            tma_load_2d_pair(sa + j * 64 * BK * 2, ta, a0 + 64 * j, k0, fb);
        } else {
          tma_load_2d_pair(sa, ta, k0, a0, fb);
        }
        const bool second = g.b_dual == 2 && kb >= g.k_split_kb;
        const CUtensorMap* tbk = second ? tb2 : tbn;
        const int kq = second ? k0 - g.k_split_kb * BK : k0;
        if (B_MN) {
#pragma unroll
          for (int j = 0; j < BM / 64; ++j)
            tma_load_2d_pair(sb + j * 64 * BK * 2, tbk, b0 + 64 * j, kq, fb);
        } else {
          tma_load_2d_pair(sb, tbk, kq, b0, fb);
        }
        ++issued;
        if (++stage == STAGES2) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        if (leader) wave_arrive(g);
        ++step;
      }
    }
  }
  if (leader) wave_finish(g, step);
  // Drain: the leader's full barriers count both CTAs' copies; once they
  // have all completed no copy of either CTA is still in flight.
  if (leader) {
    for (int s = 0; s < STAGES2; ++s) {
      const uint32_t cnt = issued / STAGES2 +
                           (static_cast<uint32_t>(s) < issued % STAGES2 ? 1u : 0u);
      if (cnt) mbar_wait(sm.full(s), (cnt - 1u) & 1u, ctx, false);
    }
  }
}

template <bool A_MN, bool B_MN>
__device__ __forceinline__ void role_mma_pair(const GemmGeom& g,
                                              const SmemMap2& sm,
                                              uint32_t tmem_base,
                                              const WaitCtx& ctx) {
  constexpr uint32_t IDESC = idesc_pair_bf16_f32<A_MN, B_MN>();
  constexpr uint32_t MN_LBO = 64 * BK * 2;
  const int nclusters = gridDim.x >> 1;
  const int cluster = blockIdx.x >> 1;
  uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
  bool ok = true;
  for (int u = cluster; ok && u < g.num_units; u += nclusters) {
    const Unit t = decode_unit(g, u, 2 * BM, 0);
    for (int tt = 0; ok && tt < t.n_count; ++tt) {
      if (!mbar_wait(sm.tempty(acc), acc_phase ^ 1u, ctx, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + acc * BN;
      for (int kb = 0; kb < g.num_kb; ++kb) {
        if (!mbar_wait(sm.full(stage), phase, ctx, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = sm.a + stage * A2_STAGE_BYTES;
        const uint32_t sb = sm.b + stage * B2_STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t ad = A_MN ? sdesc_sw128(sa + k * 2048, MN_LBO, 1024)
                                   : sdesc_sw128(sa + k * 32, 16, 1024);
          const uint64_t bd = B_MN ? sdesc_sw128(sb + k * 2048, MN_LBO, 1024)
                                   : sdesc_sw128(sb + k * 32, 16, 1024);
          tc_mma_pair(d, ad, bd, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit_pair_both(sm.empty(stage));
        if (++stage == STAGES2) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit_pair_both(sm.tfull(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  tc_commit_pair_local(sm.drain());
  mbar_wait(sm.drain(), 0, ctx, false);
}

template <class Epi>
__device__ __forceinline__ void role_epilogue_pair(
    const GemmGeom& g, const typename Epi::Params& p, const SmemMap2& sm,
    uint32_t tmem_base, uint32_t rank, const WaitCtx& ctx, int warp,
    int lane, const CUtensorMap* te, uint32_t stage_base) {
  const int q = warp & 3;
  const int r = q * 32 + lane;
  const int nclusters = gridDim.x >> 1;
  const int cluster = blockIdx.x >> 1;
  uint32_t acc = 0, acc_phase = 0;
  Epi epi;
  epi.te = te;
  epi.stage = stage_base + static_cast<uint32_t>(q) * 2u * EPI_BUF_BYTES;
  for (int u = cluster; u < g.num_units; u += nclusters) {
    const Unit t = decode_unit(g, u, 2 * BM, static_cast<int>(rank));
    epi.begin_unit(p, g, t, r);
    bool ok = true;
    for (int tt = 0; tt < t.n_count; ++tt) {
      const bool got = mbar_wait(sm.tfull(acc), acc_phase, ctx, true);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      epi.tile(p, g, t, t.n_first + tt, taddr, r);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(sm.tempty(acc), 0));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) break;
    epi.end_unit(p, g, t, r);
  }
  // every TMA store of this warp has finished reading shared memory and
  // writing global memory before the CTA may exit
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

template <class Epi, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap ta,
                const __grid_constant__ CUtensorMap tb,
                const __grid_constant__ CUtensorMap tb2, const GemmGeom g,
                const __grid_constant__ typename Epi::Params p,
                unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  SmemMap2 sm;
  sm.a = base;
  sm.b = base + STAGES2 * A2_STAGE_BYTES;
  sm.bars = base + STAGES2 * STAGE2_BYTES;
  uint8_t* misc = smem_raw + (sm.bars - raw) + 8 * (2 * STAGES2 + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(sm.full(s), 1);
      mbar_init(sm.empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(sm.tfull(a), 1);
      mbar_init(sm.tempty(a), 8);  // 4 epilogue warps x 2 CTAs
    }
    mbar_init(sm.drain(), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&ta);
    tma_prefetch_desc(&tb);
    if (g.b_dual) tma_prefetch_desc(&tb2);
  }
  // Both CTAs' barriers exist before either CTA signals the other's.
  cluster_sync_all();
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx ctx{abort_flag, err, g.timeout_ns};

  if (warp == 0) {
    if (lane == 0)
      role_producer_pair<A_MN, B_MN>(&ta, &tb, &tb2, g, sm, rank, ctx);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) role_mma_pair<A_MN, B_MN>(g, sm, tmem_base, ctx);
    __syncwarp();
  } else {
    role_epilogue_pair<Epi>(g, p, sm, tmem_base, rank, ctx, warp, lane, &tb2,
                            base + STAGES2 * STAGE2_BYTES + 1024);
  }

  tc_fence_before();
  __syncthreads();
  // Neither CTA frees its shared memory or tensor memory while the pair's
  // MMAs or the peer's barrier traffic may still touch it.
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

constexpr int GEMM2_SMEM_BYTES =
    1024 + STAGES2 * STAGE2_BYTES + 1024 + EPI_STAGE_BYTES;

template <class Epi, bool A_MN, bool B_MN>
cudaError_t launch_gemm_pair_t(const CUtensorMap& ta, const CUtensorMap& tb,
                               const GemmGeom& g,
                               const typename Epi::Params& p, unsigned* err,
                               int grid, cudaStream_t s,
                               const CUtensorMap* tb2 = nullptr) {
  auto kern = k_gemm_pair<Epi, A_MN, B_MN>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM2_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = GEMM2_SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2 ? *tb2 : tb, g, p, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace lce
