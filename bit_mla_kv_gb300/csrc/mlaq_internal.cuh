// Internal definitions shared by the libmlaq kernels and the C-ABI layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mlaq.h"

namespace mlaq {

constexpr int kPage = 64;        // tokens per page
constexpr int kSink = 4;         // sink tokens kept in BF16
constexpr int kRecent = 128;     // recent tokens kept in BF16
constexpr int kRing = kSink + kRecent;
constexpr int kDL = 512;         // content latent width
constexpr int kDR = 64;          // RoPE key width
constexpr int kD = kDL + kDR;    // 576
constexpr int kGroup = 64;       // quantization group
constexpr int kGroups = kD / kGroup;  // 9 (8 content + 1 RoPE)
constexpr int kMetaTok = kGroups * 4;  // bytes of (scale, min) fp16 pairs per token
constexpr int kMetaPage = kPage * kMetaTok;  // 2304

// Workspace layout (bytes from the workspace base).
constexpr size_t kWsStatus = 0;          // int32 sticky status
constexpr size_t kWsNumItems = 4;        // int32 number of work items of the last plan
constexpr size_t kWsAppendDone = 8;      // uint32 CTAs of the running append that have finished
constexpr int kMaxPlanCtas = 1024;       // decode CTA count never exceeds this
constexpr int kMaxSeqs = 16384;          // sequences per call
constexpr int kMaxHeadBlocks = 8;        // 128 heads / 16
// Split partial rows the plan may add beyond one per (sequence, head): the
// decode caps its item slots per head block at kPlanRowSlack / H.
constexpr int kPlanRowSlack = 32 * kMaxPlanCtas;

__host__ __device__ constexpr int content_bits(int mode) { return mode == MLAQ_C2R4 ? 2 : 4; }
// Bytes of codes per token in a page (BF16 mode: the raw token).
__host__ __device__ constexpr int token_bytes(int mode) {
  return mode == MLAQ_BF16 ? kD * 2 : (kDL * content_bits(mode) + kDR * 4) / 8;
}
__host__ __device__ constexpr int group_code_bytes(int bits) { return kGroup * bits / 8; }
__host__ __device__ constexpr int page_code_bytes(int mode) { return kPage * token_bytes(mode); }

// A work item of the split-KV decode: units [u_lo, u_hi) of sequence b,
// processed by CTA `cta`. A sequence's units are its ring chunks (16 BF16
// sink/recent slots each; packed modes) followed by its packed pages (4 units
// = 4 steps of 16 tokens each) or, in BF16 mode, 16-token quarter pages.
struct __align__(16) Item {
  int b, u_lo, u_hi, cta;
  int L, pad0, pad1, pad2;  // L: the sequence's (clamped) length when the plan was made
};

// Upper bounds of the planner's per-sequence cost (32-bit prefix sums): per
// page of a sequence, and for its ring plus item overhead.
constexpr int kPlanCostPerPage = 32, kPlanCostRingMax = 512;
// Default planning costs (see the planner): packed step, ring step, item start.
constexpr int kDefCostStep = 8, kDefCostRing = 19, kDefCostItem = 40;
inline bool plan_cost_fits(int max_seqs, int max_pages_per_seq) {
  return (long long)max_seqs * ((long long)max_pages_per_seq * kPlanCostPerPage + kPlanCostRingMax) < 0x7fffffffLL;
}

// Items: at most one per sequence plus one per CTA boundary inside a sequence.
inline size_t max_items_for(int max_seqs) { return (size_t)max_seqs + kMaxPlanCtas + 1; }
// Rows (item, head) of the partial outputs. A plan over G item slots has at
// most B + G + 1 items, and G <= kPlanRowSlack / H, so items * H <= B H +
// kPlanRowSlack + H.
inline size_t max_partial_rows(int max_seqs, int max_heads) {
  return (size_t)max_seqs * max_heads + (size_t)kPlanRowSlack + max_heads;
}
// Item slots (CTAs per head block) of a decode over H heads in HB head blocks
// with `ctas` CTAs in all: the planner's one-pass scan over slot boundaries
// needs G + 1 <= kMaxPlanCtas, and the partial rows need G * H <= kPlanRowSlack.
inline int plan_slots(int ctas, int HB, int H) {
  int G = ctas / HB;
  if (G > kMaxPlanCtas - 1) G = kMaxPlanCtas - 1;
  if (G > kPlanRowSlack / H) G = kPlanRowSlack / H;
  return G < 1 ? 1 : G;
}

struct WsLayout {
  size_t items, item_start, cta_first, cta_item_start, lse_part, o_part, total;
};
inline WsLayout ws_layout(int max_seqs, int max_heads) {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  WsLayout L;
  size_t off = 256;
  L.items = off;          off += al(max_items_for(max_seqs) * sizeof(Item));
  L.item_start = off;     off += al(((size_t)max_seqs + 1) * 4);
  L.cta_first = off;      off += al(((size_t)kMaxPlanCtas + 1) * sizeof(Item));
  L.cta_item_start = off; off += al(((size_t)kMaxPlanCtas + 1) * 4);
  const size_t rows = max_partial_rows(max_seqs, max_heads);
  L.lse_part = off;       off += al(rows * 4);
  L.o_part = off;         off += rows * kDL * 2;  // fp16 partial outputs
  L.total = off;
  return L;
}

// BF16 rows (ring slots, BF16-mode page tokens): element position of channel
// e in row r; the 16-byte chunks are XOR-permuted by r mod 8.
__host__ __device__ inline int bf16_row_pos(int e, int r) { return (((e >> 3) ^ (r & 7)) << 3) | (e & 7); }

// ---------------------------------------------------------------------------
// Physical code layout inside a token's bytes.
//
// Per token: content groups g = 0..7 (32 B each for INT4, 16 B for INT2), then
// the RoPE group (32 B, INT4). The channel order inside a group is permuted so
// that one 64-bit (INT4) or 32-bit (INT2) shared-memory load gives a thread
// exactly the fp16 pairs of the m16n8k16 B fragments it needs, and so that
// a LOP3 with a 0x6400 exponent turns two codes into an fp16 pair (1024 + m*q)
// without shifts. The canonical order (code i of the segment in bits
// [b*(i mod k), +b) of byte i/k) is produced by mlaq_export_tokens.
//
// Shared notation: for channel c of a 64-channel group,
//   kk = c >> 4 (MMA k-step), bi = (c >> 3) & 1 (B register b0/b1),
//   i = (c >> 1) & 3 (thread in the quad), ln = c & 1 (fp16 lane in the pair).
// Returns the bit offset of the code inside the group's bytes.
__host__ __device__ constexpr int content_code_bit(int c, int bits) {
  int kk = c >> 4, bi = (c >> 3) & 1, i = (c >> 1) & 3, ln = c & 1;
  if (bits == 4) {
    int word = 2 * i + (kk >> 1);
    int p = 2 * (kk & 1) + bi;  // 0: bits 0-3, 1: 4-7, 2: 8-11, 3: 12-15 of each 16-bit lane
    return word * 32 + 16 * ln + 4 * (p & 1) + 8 * (p >> 1);
  } else {
    int word = i;
    int p = 2 * kk + bi;  // 0..7: 2-bit field (p & 3) of byte (p >> 2) of each 16-bit lane
    return word * 32 + 16 * ln + 2 * (p & 3) + 8 * (p >> 2);
  }
}
// RoPE group (INT4): warp w of the decode kernel owns k-step kk = w.
__host__ __device__ constexpr int rope_code_bit(int c) {
  int kk = c >> 4, bi = (c >> 3) & 1, i = (c >> 1) & 3, ln = c & 1;
  int word = 2 * kk + (i >> 1);
  return word * 32 + 16 * ln + 8 * (i & 1) + 4 * bi;
}

// ---------------------------------------------------------------------------
// PTX helpers.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Programmatic dependent launch: wait for the grid this one depends on (a
// no-op when launched without the attribute), and let the next grid launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// try_wait that may suspend the thread for up to `hint_ns` until the phase
// completes (no spinning on the issue slots of the SM sub-partition).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Bounded wait: returns false if the phase did not complete within
// `limit_ns` nanoseconds of wall time (a try_wait may suspend the thread, so
// the bound is on time, not on the number of polls).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// The same bound, with suspending polls (for waits that are often long).
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// Bulk (TMA) copy global -> shared, completion signalled on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Barrier that also ORs a predicate across the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

// Pure register operations: not volatile, so independent ones can be
// interleaved by the compiler.
// Four 8x8 b16 matrices from shared memory in the mma fragment layout; lane
// L gives the 16-byte row address of row L % 8 of matrix L / 8.
__device__ __forceinline__ void ldmatrix_x4(uint32_t saddr, uint32_t (&f)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(f[0]), "=r"(f[1]), "=r"(f[2]), "=r"(f[3])
               : "r"(saddr)
               : "memory");
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
// D += A * B, m16n8k16, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }


// ---------------------------------------------------------------------------
// tcgen05 / tensor memory (TMEM) helpers. TMEM addresses: bits 31..16 lane,
// bits 15..0 column. A warp may only touch the 32-lane quadrant
// [32 (warp % 4), +32).
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish() {  // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 lanes x 256 bits: thread t writes lanes (t/4, t/4 + 8), columns (2 (t%4), 2 (t%4) + 1)
__device__ __forceinline__ void tmem_st_16x256b(uint32_t taddr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r0), "r"(r1), "r"(r2),
               "r"(r3)
               : "memory");
}
// Four 16x256b tiles side by side (columns 0-7, 8-15, 16-23, 24-31): regs
// 4k..4k+3 go to column block k in the x1 layout.
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// 32 lanes x 32 bits x 16: thread t reads lane t, 16 consecutive columns
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// 32 lanes x 32 bits x 32 columns: thread t stores / loads lane t.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// Shared-memory matrix descriptor, no swizzle: 8-row x 16-byte core matrices;
// k_stride = bytes between cores adjacent along K, mn_stride = along M/N.
__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t saddr, uint32_t k_stride, uint32_t mn_stride) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((k_stride >> 4) & 0x3FFFu) << 16;   // leading-dimension byte offset
  d |= (uint64_t)((mn_stride >> 4) & 0x3FFFu) << 32;  // stride-dimension byte offset
  d |= (uint64_t)1 << 46;                              // descriptor version
  return d;
}
// Instruction descriptor, kind::f16: fp16 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same with bf16 A and B (both operands always share one type).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return umma_idesc_f16(M, N) | (1u << 7) | (1u << 10);
}
// D (TMEM) (+)= A (TMEM) x B (smem descriptor)^T; issued by one thread.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_t, uint32_t a_t, uint64_t bdesc, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_t),
      "r"(a_t), "l"(bdesc), "r"(idesc), "r"((uint32_t)acc)
      : "memory");
}
// mbarrier arrive once all tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_view_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
}  // namespace mlaq

// Host-side handle.
struct mlaq_cache {
  int mode;
  int32_t num_pages, max_seqs, max_pages_per_seq, max_heads;
  void* codes;
  void* meta;
  void* ring;
  void* workspace;
  size_t workspace_bytes;
  int num_sms;
  int decode_ctas;
  int decode_ctas_set;  // decode_ctas chosen by mlaq_set_decode_ctas
  int decode_variant;   // mlaq_set_decode_variant: 0 auto, 1 register scores, 2 tcgen05 scores
  int cost_step, cost_ring, cost_item;  // planner costs (mlaq_set_plan_costs)
  // timing
  int timing_max;
  int timing_n;
  void** timing_events;  // cudaEvent_t pairs
};

// Kernel launchers (defined in the .cu files).
namespace mlaq {
cudaError_t launch_append(const mlaq_cache* c, const int32_t* page_table, int32_t* seq_lens, int B,
                          const uint16_t* c_latent, const uint16_t* k_rope, int n_new, const int32_t* cu_new,
                          int total_new, cudaStream_t s);
cudaError_t launch_export(const mlaq_cache* c, const int32_t* page_table, int B, const int32_t* token_b,
                          const int32_t* token_t, int n, uint8_t* codes_out, uint16_t* meta_out, cudaStream_t s);
cudaError_t launch_decode(mlaq_cache* c, const uint16_t* q_latent, const uint16_t* q_rope,
                          const int32_t* page_table, const int32_t* seq_lens, int B, int H, float scale,
                          uint16_t* out, float* lse, cudaStream_t s, int q_len = 1);
}  // namespace mlaq
