// Split-KV MLA decode over the mixed-precision paged cache: a device planner,
// a persistent attention kernel and a log-sum-exp combine kernel.
//
// QuantMLA (ai.info "Key Contributions" item 4; onedev.kr "어떻게 쓰나"):
// unpack + dequant fused into attention, packed pages and metadata staged
// apart from the reconstructed tiles, 4 sink + 128 recent tokens read from
// BF16, a single softmax over all valid tokens.
//
// Work distribution. A sequence's work is a list of units: its 9 ring chunks
// (16 BF16 sink/recent slots each) and then its packed pages (4 units each,
// one per 16-token sub-step); in the all-BF16 cache a unit is a 16-token
// quarter page. The planner gives each of the G persistent CTAs of a head
// block an equal share of the concatenated unit list by a cost model, cut at
// page boundaries. The share of one CTA inside one sequence is a work item;
// a sequence with one item is finalized by the attention kernel, otherwise
// the combine kernel merges its items' normalized partials.
//
// Attention (one CTA = NH = 16 or 32 heads, 4 warps; three 16-head or two
// 32-head CTAs per SM):
//  * Pages (codes + fp16 meta) or ring chunks are staged by bulk copies
//    (TMA) into a 2-stage shared-memory ring per CTA that runs ahead across
//    items; every wait is bounded in wall time.
//  * A packed page is one body of four 16-token sub-steps (32-head CTAs) or
//    two bodies of two (16-head CTAs), each under one pair of barriers; ring
//    chunks and BF16 page quarters are 16-token steps.
//  * Warp w owns content groups 2w, 2w+1 (channels 128w..128w+127) and RoPE
//    channels 16w..16w+15.
//  * Scores use exact integer codes as fp16 MMA operands: per group g,
//    D_g[t,h] = sum_{c in g} q[t,c] Q[h,c], then
//    S[t,h] = sum_g s[t,g] D_g[t,h] + sum_g mn[t,g] sum_{c in g} Q[h,c]
//    (the second sum is one more m16n8k16 MMA on hi/lo fp16 splits of the
//    per-group query sums): exact up to fp32 rounding. A 32-head CTA runs
//    this per 16-head half on the same unpacked codes.
//  * The four warps' partial scores meet in shared memory; each thread runs
//    the online softmax for one head (exp2, lazily rescaled max) and writes
//    P^T in fp16 as the B operand of the aggregation.
//  * Aggregation on tcgen05: the codes are dequantized once to fp16 (q*s +
//    mn, one rounding), transposed in registers with movmatrix and stored to
//    TMEM (lanes = channels); one tcgen05.mma per sub-step and channel block
//    accumulates O^T += V^T P^T in TMEM while the warps unpack the next page.
//  * BF16 ring tokens of a packed cache take the same path with
//    (s, mn) = (1, 0); an all-BF16 cache runs both contractions on its bf16
//    values as given (bf16 register MMAs for the scores, bf16 tcgen05
//    operands for the aggregation).
#include <math.h>

#include <atomic>
#include <mutex>

#include "mlaq_internal.cuh"

namespace mlaq {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kT = 16;                                // tokens per step
constexpr int kRingChunks = (kRing + kT - 1) / kT;    // 9
constexpr int kStageBytes = kPage * 288 + kMetaPage;  // 20736: max(C4R4 page + meta, 16 BF16 tokens)
constexpr uint64_t kWaitLimit = 200000000ull;  // 200 ms per bounded wait
constexpr int kMaxDevices = 64;
template <bool B>
struct BoolC {
  static constexpr bool value = B;
};
// floats per row of partial scores [h][t]: 64 tokens of a page step + 4 (bank spread)
// Per head count: a packed page is processed in 4 / subs bodies of `subs`
// 16-token sub-steps each (one pair of barriers and one softmax per body).
// 16-head CTAs take half pages: their TMEM (O^T 64 columns + A 64) and
// shared memory (2 stages, 32-token score tiles) fit three CTAs per SM at 168
// registers, which measured faster than whole pages at two CTAs per SM
// (V2-Lite C4R4 110.4 vs 115.7 us per call). 32-head CTAs keep whole pages
// at two per SM (O^T alone takes 128 columns).
// (Measured alternatives for 16-head CTAs on V2-Lite C4R4: four per SM at 128
// registers, 60 bytes of spills: 117.5 us; three stages: 111.8 us; against
// 110.5 us for three per SM, 168 registers, two stages.)
template <int NH>
__host__ __device__ constexpr int body_subs() { return NH == 16 ? 2 : 4; }
template <int NH>
__host__ __device__ constexpr int ctas_per_sm() { return NH == 16 ? 3 : 2; }
template <int NH>
__host__ __device__ constexpr int sp_stride() { return 16 * body_subs<NH>() + 4; }  // floats per score row
// Aggregation on tcgen05: O^T[channel][head] accumulates in TMEM.
constexpr int kAggBufs = 2;      // A (content) / P^T step buffers in flight
// TMEM columns of a CTA: O^T (4 blocks x NH heads), then A (sub-steps x 4 blocks x 8 columns)
template <int NH>
__host__ __device__ constexpr uint32_t tmem_cols() { return 4 * NH + 32 * body_subs<NH>() <= 128 ? 128 : 256; }
// first TMEM column of the A step buffers for NH heads per CTA
template <int NH>
__host__ __device__ constexpr uint32_t tmem_a_col() { return 4 * NH; }

struct DecodeParams {
  const uint8_t* codes;
  const uint8_t* meta;
  const uint16_t* ring;
  const uint16_t* q_latent;
  const uint16_t* q_rope;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int* status;
  const Item* items;
  const int* item_start;
  const int* cta_item_start;
  const Item* cta_first;  // first item of each CTA; pad0 = page of its first stage
  __half* o_part;  // normalized split partials, fp16
  float* lse_part;
  uint16_t* out;
  float* lse;
  int B, H, HB, max_pages, num_pages, max_tokens;
  int q_len, h_per_q;  // query tokens per sequence; heads per query token (H = q_len * h_per_q)
  int cost_step, cost_ring, cost_item;  // planning costs
  float scale_log2;
  // CTA shares by dispatch slot (linear CTA index / SMs): relative speeds x
  // 1000 of the first, second and third CTA resident on an SM
  int sms, slot_w[3];
};

// Shared memory of a decode CTA serving NH heads (16, or 32 when H is a
// multiple of 32: the two 16-head halves then share every page's unpack; the
// larger score and P tiles and the second half's query fragments leave room
// for two stages at two CTAs per SM).
template <int NH>
struct __align__(128) DecodeSmem {
  static constexpr int kNumStages = 2;
  static constexpr int kQxWords = NH == 16 ? 1 : 10 * kThreads;  // 38 fragment words per thread, as uint4
  uint8_t stage[kNumStages][kStageBytes];
  float sp[kWarps][NH][sp_stride<NH>()];  // partial scores, [warp][head][token]
  float alpha[NH];
  float fin_m[NH];
  float fin_l[NH];
  int stage_bad[kNumStages];
  uint64_t full[kNumStages];
  __align__(128) uint8_t pt[kAggBufs][32 * NH];  // P^T B operand: NH heads x 16 tokens, 8x8 core matrices
  __align__(128) uint8_t ptp[body_subs<NH>()][32 * NH];  // P^T of the sub-steps of a page body
  uint64_t agg_done[kAggBufs];
  uint32_t tmem_base;
  int rescale_flag[kWarps];
  uint4 qx[kQxWords];  // query fragments of heads 16..31 of the block, [word / 4][thread]
};
// ctas_per_sm CTAs per SM: 228 KB of shared memory, 1 KB of it reserved per CTA
static_assert(sizeof(DecodeSmem<16>) * ctas_per_sm<16>() + 1024 * ctas_per_sm<16>() <= 228 * 1024 &&
                  sizeof(DecodeSmem<32>) * ctas_per_sm<32>() + 1024 * ctas_per_sm<32>() <= 228 * 1024,
              "decode shared memory must allow ctas_per_sm CTAs per SM");
static_assert(tmem_cols<16>() * ctas_per_sm<16>() <= 512 && tmem_cols<32>() * ctas_per_sm<32>() <= 512,
              "decode TMEM must allow ctas_per_sm CTAs per SM");
// the page-body softmax reads its tokens four at a time (2 * subs per thread)
static_assert((body_subs<16>() == 2 || body_subs<16>() == 4) && (body_subs<32>() == 2 || body_subs<32>() == 4),
              "page bodies of two or four sub-steps");

__device__ __forceinline__ int clamp_len(int L, int max_tokens) { return min(max(L, 0), max_tokens); }
// Units of a sequence and its leading ring units.
__device__ __forceinline__ int ring_units(int mode, int L) { return (mode != MLAQ_BF16 && L > 0) ? kRingChunks : 0; }
__device__ __forceinline__ int seq_units(int mode, int L) {
  if (mode == MLAQ_BF16) return (L + kT - 1) / kT;
  const int pages = L > kRing ? (L - kRecent + kPage - 1) / kPage : 0;
  return ring_units(mode, L) + 4 * pages;
}
// Planning cost (DecodeParams cost_*), by default in eighths of a packed
// step (16 tokens) as measured on GB300: a packed or BF16-page step costs 8;
// a ring step 19 (its BF16 tile runs 16 tokens per barrier pair, packed
// pages 64: 3300 against 1370 cycles per 16 tokens); the first ring unit of a
// sequence carries 40 more for the item switch (query load, epilogue) of the
// CTA that starts it. The host keeps 4 * step <= kPlanCostPerPage and
// item + 9 * ring <= kPlanCostRingMax, the bounds of its overflow check.
static_assert(4 * kDefCostStep <= kPlanCostPerPage && kDefCostItem + kDefCostRing * kRingChunks <= kPlanCostRingMax,
              "planner cost bounds");
__device__ __forceinline__ int ring_cost(const DecodeParams& p, int R) {
  return R > 0 ? p.cost_item + p.cost_ring * R : 0;
}
__device__ __forceinline__ int seq_cost(const DecodeParams& p, int mode, int L) {
  const int R = ring_units(mode, L);
  return ring_cost(p, R) + p.cost_step * (seq_units(mode, L) - R);
}
// Unit index of a cost offset inside a sequence that lies on a unit boundary.
__device__ __forceinline__ int cost_to_unit(const DecodeParams& p, int mode, int L, int x) {
  const int R = ring_units(mode, L);
  const int xr = ring_cost(p, R);
  if (x >= xr) return R + (x - xr) / p.cost_step;
  return x < p.cost_item + p.cost_ring ? 0 : (x - p.cost_item) / p.cost_ring;
}

// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32).
__device__ int block_excl_scan(int v, int* red, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += u;
  }
  __syncthreads();
  if (lane == 31) red[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int y = lane < (int)(blockDim.x >> 5) ? red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += u;
    }
    red[lane] = y;
  }
  __syncthreads();
  const int warp_prefix = wid ? red[wid - 1] : 0;
  *total = red[31];
  return warp_prefix + x - v;
}

// Weighted count of the item slots below c. Item slot c' of head block x is
// linear CTA c' * HB + x, dispatched round-robin over the SMs, so it is the
// (c' * HB / sms)-th CTA resident on its SM. The CTAs that share an SM run at
// different speeds (the warps of the CTA dispatched first are scheduled
// first): each gets a share of the cost in proportion to its slot's speed.
__device__ __forceinline__ long long slot_weight_below(const DecodeParams& p, int c) {
  long long w = 0;
  int lo = 0;
  for (int k = 0; k < 3; ++k) {
    const int hi = k == 2 ? c : min(c, (int)(((long long)(k + 1) * p.sms + p.HB - 1) / p.HB));
    if (hi > lo) w += (long long)(hi - lo) * p.slot_w[k];
    lo = max(lo, hi);
  }
  return w;
}

// Largest index i in [lo, hi] with a[i] <= key (a non-decreasing, a[lo] <= key).
__device__ __forceinline__ int last_le(const int* a, int lo, int hi, int key) {
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= key) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Planner: one CTA of 1024 threads, on the device (no host sync). Its working
// arrays live in dynamic shared memory, so no pass waits on dependent
// global-memory loads: useq[B+1] (unit prefix), sitem[B+1] (first item of
// each sequence), bnd[G+1] (CTA boundaries), ne[G+1] (non-empty CTAs below).
__host__ __device__ inline size_t plan_smem_bytes(int B, int G) {
  return (size_t)(2 * (B + 1) + 2 * (G + 1)) * sizeof(int);
}
// Page-table entry of an item's first stage (0 for a ring chunk, -1 when the
// page index is outside the table).
__device__ __forceinline__ int first_stage_page(const DecodeParams& p, int mode, const Item& it) {
  int pidx;
  if (mode == MLAQ_BF16) {
    pidx = it.u_lo / 4;
  } else {
    const int R = ring_units(mode, it.L);
    if (it.u_lo < R) return 0;
    pidx = (it.u_lo - R) / 4;
  }
  return pidx < p.max_pages ? p.page_table[(size_t)it.b * p.max_pages + pidx] : -1;
}

__global__ void __launch_bounds__(1024) plan_kernel(DecodeParams p, int mode, int G, Item* items, int* item_start,
                                                    int* cta_item_start, Item* cta_first, int* num_items) {
  extern __shared__ int plan_smem[];
  __shared__ int red[32];
  __shared__ int carry_s;
  pdl_wait();               // seq_lens may come from the kernel before
  pdl_launch_dependents();  // the decode grid may launch and wait for this one
  const int tid = threadIdx.x;
  const int B = p.B;
  int* useq = plan_smem;       // [B + 1] cost prefix
  int* sfc = useq + (B + 1);    // [B + 1] first item << 10 | first CTA of each sequence
  int* bnd = sfc + (B + 1);     // [G + 1] CTA boundaries (cost)
  int* ne = bnd + (G + 1);      // [G + 1] non-empty CTAs below c
  // A: units per sequence -> useq (exclusive prefix); reset the merge
  //    empty sequences get out = 0, lse = -inf.
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + tid;
    int u = 0;
    if (b < B) {
      const int Lraw = p.seq_lens[b];
      if (Lraw > p.max_tokens) atomicOr(p.status, MLAQ_DEV_SEQ_OVERFLOW);
      const int L = clamp_len(Lraw, p.max_tokens);
      u = seq_cost(p, mode, L);
      if (L == 0) {
        for (int k = 0; k < p.H * kDL; ++k) p.out[(size_t)b * p.H * kDL + k] = 0;
        for (int h = 0; h < p.H; ++h) p.lse[(size_t)b * p.H + h] = -INFINITY;
      }
    }
    int tot;
    const int ex = block_excl_scan(u, red, &tot);
    const int carry = carry_s;
    if (b < B) useq[b] = carry + ex;
    __syncthreads();
    if (tid == 0) carry_s = carry + tot;
    __syncthreads();
  }
  if (tid == 0) useq[B] = carry_s;
  __syncthreads();
  const int U = useq[B];
  // B: CTA boundaries (in cost): the slot-weighted share of c, snapped down
  //    to a step start, and to a page start inside packed pages.
  const long long w_all = slot_weight_below(p, G);
  for (int c = tid; c <= G; c += blockDim.x) {
    const int raw = c >= G ? U : (int)(((long long)U * slot_weight_below(p, c)) / w_all);
    int v = raw;
    if (raw < U) {
      const int b = last_le(useq, 0, B, raw);
      const int R = ring_units(mode, clamp_len(p.seq_lens[b], p.max_tokens));
      const int xr = ring_cost(p, R);
      int x = raw - useq[b];
      const int cs = p.cost_step, cr = p.cost_ring, ci = p.cost_item;
      if (x < xr)
        x = x < ci + cr ? 0 : ci + ((x - ci) / cr) * cr;
      else
        x = xr + ((x - xr) / (mode == MLAQ_BF16 ? cs : 4 * cs)) * (mode == MLAQ_BF16 ? cs : 4 * cs);
      v = useq[b] + x;
    }
    bnd[c] = v;
  }
  __syncthreads();
  // C: ne[c] = number of non-empty CTAs below c (G + 1 <= 1024)
  {
    const int c = tid;
    const int nonempty = (c < G && bnd[c] < bnd[c + 1]) ? 1 : 0;
    int tot;
    const int ex = block_excl_scan(nonempty, red, &tot);
    if (c <= G) ne[c] = ex;
    __syncthreads();
  }
  // D: item counts per sequence (one per non-empty CTA overlapping it) ->
  //    first item of each sequence (exclusive prefix)
  if (tid == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + tid;
    int cnt = 0, c_lo = 0;
    if (b < B) {
      const int u0 = useq[b], u1 = useq[b + 1];
      if (u1 > u0) {
        c_lo = last_le(bnd, 0, G - 1, u0);
        const int c_hi = last_le(bnd, 0, G - 1, u1 - 1);
        cnt = ne[c_hi + 1] - ne[c_lo];
      }
    }
    int tot;
    const int ex = block_excl_scan(cnt, red, &tot);
    const int carry = carry_s;
    if (b < B) {
      item_start[b] = carry + ex;
      sfc[b] = ((carry + ex) << 10) | c_lo;  // items < 2^21, CTAs < 2^10
    }
    __syncthreads();
    if (tid == 0) carry_s = carry + tot;
    __syncthreads();
  }
  const int n = carry_s;
  if (tid == 0) {
    item_start[B] = n;
    *num_items = n;
  }
  // E: one thread per CTA writes its items. Items are ordered by sequence,
  // then CTA: the item of (sequence b, CTA c) is sitem[b] plus the non-empty
  // CTAs between the first CTA of b and c. An empty CTA gets the index of the
  // next item, so its item range is empty.
  for (int c = tid; c <= G; c += blockDim.x) {
    int v = n;
    if (bnd[c] < U) {
      const int bs = last_le(useq, 0, B, bnd[c]);
      v = (sfc[bs] >> 10) + ne[c] - ne[sfc[bs] & 1023];
      if (c < G && bnd[c] < bnd[c + 1]) {
        int k = v;
        for (int b = bs; b < B && useq[b] < bnd[c + 1]; ++b) {
          const int u0 = useq[b], u1 = useq[b + 1];
          if (u1 == u0) continue;  // empty sequence: no item
          const int Lb = clamp_len(p.seq_lens[b], p.max_tokens);
          const Item it{b, cost_to_unit(p, mode, Lb, max(bnd[c], u0) - u0), cost_to_unit(p, mode, Lb, min(bnd[c + 1], u1) - u0),
                        c, Lb, 0, 0, 0};
          items[k] = it;
          if (k == v) {
            // the CTA's first item, with the page of its first stage, so that
            // the decode CTA can issue its first copy after a single load
            Item f = it;
            f.pad0 = first_stage_page(p, mode, f);
            cta_first[c] = f;
          }
          ++k;
        }
      }
    }
    cta_item_start[c] = v;
  }
}

// ---------------------------------------------------------------------------
// Unpack helpers: fp16 pair (1024 + m*q) via LOP3, then exact q via HFMA2.
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, uint32_t mask, uint32_t inv_m, uint32_t neg_off) {
  uint32_t v = lop3_and_or(w, mask, 0x64006400u);
  return h2_as_u32(__hfma2(u32_as_h2(v), u32_as_h2(inv_m), u32_as_h2(neg_off)));
}
// fp16 constants as packed pairs
constexpr uint32_t kH1 = 0x3C003C00u;      // 1.0
constexpr uint32_t kHm1024 = 0xE400E400u;  // -1024
constexpr uint32_t kH1_4 = 0x34003400u;    // 0.25
constexpr uint32_t kHm256 = 0xDC00DC00u;   // -256
constexpr uint32_t kH1_16 = 0x2C002C00u;   // 0.0625
constexpr uint32_t kHm64 = 0xD400D400u;    // -64
constexpr uint32_t kH1_64 = 0x24002400u;   // 0.015625
constexpr uint32_t kHm16 = 0xCC00CC00u;    // -16

// INT4: position p (0..3) of a word -> fp16 pair of exact codes.
__device__ __forceinline__ uint32_t int4_pos(uint32_t w, uint32_t w8, int p) {
  switch (p) {
    case 0: return unpack_pair(w, 0x000F000Fu, kH1, kHm1024);
    case 1: return unpack_pair(w, 0x00F000F0u, kH1_16, kHm64);
    case 2: return unpack_pair(w8, 0x000F000Fu, kH1, kHm1024);
    default: return unpack_pair(w8, 0x00F000F0u, kH1_16, kHm64);
  }
}
// INT2: position p (0..7) of a word.
__device__ __forceinline__ uint32_t int2_pos(uint32_t w, uint32_t w8, int p) {
  uint32_t x = p < 4 ? w : w8;
  switch (p & 3) {
    case 0: return unpack_pair(x, 0x00030003u, kH1, kHm1024);
    case 1: return unpack_pair(x, 0x000C000Cu, kH1_4, kHm256);
    case 2: return unpack_pair(x, 0x00300030u, kH1_16, kHm64);
    default: return unpack_pair(x, 0x00C000C0u, kH1_64, kHm16);
  }
}

__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t u) {
  float2 f = make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  return h2_as_u32(__float22half2_rn(f));
}
// A bf16 pair of a BF16 token as an MMA operand: converted to fp16 beside
// packed tokens (ring steps), as it is in an all-BF16 cache.
template <int MODE>
__device__ __forceinline__ uint32_t bf_operand(uint32_t u) {
  if constexpr (MODE == MLAQ_BF16)
    return u;
  else
    return bf2_to_h2(u);
}

// Ring slot validity for a sequence of length L. Slot j < 4 holds sink token
// j. Slot 4 + r holds the newest token t < L with t mod 128 == r, valid iff
// t >= 4; in closed form: r < L - 128 (then t >= 128) or 4 <= r < L (t = r).
__device__ __forceinline__ bool ring_slot_valid(int slot, int L) {
  if (slot < kSink) return slot < L;
  const int r = slot - kSink;
  return slot < kRing && ((r < L - kRecent) || (r >= kSink && r < L));
}

// Stage k of item `it` (sequence length L):
//   kind 0: ring chunk (1 step; rows are ring slots 16*idx + j)
//   kind 1: packed page (4 steps; rows are tokens 64*idx + j)
//   kind 2: BF16 quarter page (1 step; rows are tokens 16*idx + j)
struct StageRef {
  int kind, idx;
};
template <int MODE>
__device__ __forceinline__ int item_stages(const Item& it, int L) {
  if (MODE == MLAQ_BF16) return it.u_hi - it.u_lo;
  const int R = ring_units(MODE, L);
  const int n_ring = max(0, min(it.u_hi, R) - it.u_lo);
  const int n_pages = it.u_hi > R ? (it.u_hi - R) / 4 - (max(it.u_lo, R) - R) / 4 : 0;
  return n_ring + n_pages;
}
template <int MODE>
__device__ __forceinline__ StageRef item_stage(const Item& it, int L, int k) {
  if (MODE == MLAQ_BF16) return StageRef{2, it.u_lo + k};
  const int R = ring_units(MODE, L);
  const int n_ring = max(0, min(it.u_hi, R) - it.u_lo);
  if (k < n_ring) return StageRef{0, it.u_lo + k};
  return StageRef{1, (max(it.u_lo, R) - R) / 4 + (k - n_ring)};
}
// Row j of a stage holds a token that attention must see.
template <int MODE>
__device__ __forceinline__ bool row_valid(const StageRef& st, int j, int L) {
  const int t16 = kT * st.idx + j;     // ring slot (kind 0) or token (kind 2)
  const int t64 = kPage * st.idx + j;  // token (kind 1)
  const bool ring = ring_slot_valid(t16, L);
  const bool page = (t64 >= kSink) & (t64 < L - kRecent);
  const bool quarter = t16 < L;
  return st.kind == 0 ? ring : (st.kind == 1 ? page : quarter);
}

// Position of the token in row j of a stage (valid rows only): ring slot j < 4
// holds sink token j, slot 4 + r the newest token t < L with t mod 128 == r.
template <int MODE>
__device__ __forceinline__ int row_token(const StageRef& st, int j, int L) {
  if (st.kind == 1) return kPage * st.idx + j;
  const int slot = kT * st.idx + j;
  if (st.kind == 2) return slot;
  return slot < kSink ? slot : L - 1 - ((L - 1 - (slot - kSink)) % kRecent);
}

// Producer: issue the bulk copies of a stage into buffer `buf`.
template <int MODE, class SM>
__device__ void issue_stage(const DecodeParams& p, SM& sm, int b, const StageRef& st, int page, int buf) {
  uint64_t* bar = &sm.full[buf];
  if (st.kind == 0) {
    const int base = kT * st.idx;
    const int n = min(kT, kRing - base);
    const uint32_t bytes = n * kD * 2;
    sm.stage_bad[buf] = 0;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(sm.stage[buf], p.ring + ((size_t)b * kRing + base) * kD, bytes, bar);
    return;
  }
  if (page < 0 || page >= p.num_pages) {
    atomicOr(p.status, MLAQ_DEV_PAGE_OOB);
    sm.stage_bad[buf] = 1;
    mbar_arrive_expect_tx(bar, 0);
    return;
  }
  sm.stage_bad[buf] = 0;
  if constexpr (MODE == MLAQ_BF16) {
    const uint32_t bytes = kT * kD * 2;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(sm.stage[buf], p.codes + (size_t)page * page_code_bytes(MODE) + (size_t)(st.idx % 4) * bytes, bytes, bar);
  } else {
    const uint32_t cb = page_code_bytes(MODE);
    mbar_arrive_expect_tx(bar, cb + kMetaPage);
    bulk_g2s(sm.stage[buf], p.codes + (size_t)page * cb, cb, bar);
    bulk_g2s(sm.stage[buf] + cb, p.meta + (size_t)page * kMetaPage, kMetaPage, bar);
  }
}

// Page-table entry of stage k of item `it` (-1 when out of the table); ring
// chunks need none.
template <int MODE>
__device__ __forceinline__ int stage_page(const DecodeParams& p, const Item& it, int k) {
  const StageRef st = item_stage<MODE>(it, it.L, k);
  if (st.kind == 0) return 0;
  const int pidx = st.kind == 1 ? st.idx : st.idx / 4;
  return pidx < p.max_pages ? p.page_table[(size_t)it.b * p.max_pages + pidx] : -1;
}

// Producer cursor over the CTA's stage stream (all its items, in order). The
// page-table entry of the stage at the cursor and the item after the current
// one are loaded one call ahead, so issuing a stage never waits on a global
// load.
struct ProdCursor {
  int item, k, nst, issued, page;
  Item cur, nxt;
};
template <int MODE>
__device__ void producer_init(const DecodeParams& p, ProdCursor& pc, const Item& first, int i0, int i1) {
  pc.item = i0;
  pc.k = 0;
  pc.issued = 0;
  pc.cur = first;  // the planner's copy of items[i0], pad0 = page of stage 0
  pc.nst = item_stages<MODE>(pc.cur, pc.cur.L);
  if (i0 + 1 < i1) pc.nxt = p.items[i0 + 1];
  pc.page = first.pad0;
}
template <int MODE, class SM>
__device__ void producer_advance(const DecodeParams& p, SM& sm, ProdCursor& pc, int i1) {
  if (pc.item >= i1) return;
  issue_stage<MODE>(p, sm, pc.cur.b, item_stage<MODE>(pc.cur, pc.cur.L, pc.k), pc.page, pc.issued % SM::kNumStages);
  pc.issued++;
  if (++pc.k >= pc.nst) {  // items always have at least one stage
    pc.item++;
    pc.k = 0;
    if (pc.item >= i1) return;
    pc.cur = pc.nxt;
    pc.nst = item_stages<MODE>(pc.cur, pc.cur.L);
    if (pc.item + 1 < i1) pc.nxt = p.items[pc.item + 1];
  }
  pc.page = stage_page<MODE>(p, pc.cur, pc.k);
}

// Register budget of the attention kernel: 168 for three 16-head CTAs per
// SM (no spills), 240 for two 32-head CTAs (measured 1-2% faster than the 221
// registers that two CTAs per SM as launch bounds give).
template <int NH>
__host__ __device__ constexpr int decode_maxnreg() { return NH == 16 ? 168 : 240; }
template <int MODE, int NH>
__global__ void __maxnreg__(decode_maxnreg<NH>()) decode_kernel(DecodeParams p) {
  static_assert(NH == 16 || NH == 32, "16 or 32 heads per CTA");
  using SM = DecodeSmem<NH>;
  constexpr int kS = SM::kNumStages;
  constexpr int NP = NH / 16;                       // 16-head halves sharing each unpack
  constexpr uint32_t kTmemA = tmem_a_col<NH>();
  constexpr int kSubs = body_subs<NH>();      // sub-steps per page body
  constexpr int kPageParts = 4 / kSubs;        // page bodies per packed page
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int cta = blockIdx.y;
  pdl_wait();  // the plan
  pdl_launch_dependents();
  // issued together: the CTA's item range and its first item
  const Item first = threadIdx.x == 0 ? p.cta_first[cta] : Item{};
  const int i0 = p.cta_item_start[cta], i1 = p.cta_item_start[cta + 1];
  if (i0 >= i1) return;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, i = lane & 3;
  const int hb_idx = blockIdx.x;
  const int h0 = hb_idx * NH;
  const int H = p.H;
  constexpr int CB = token_bytes(MODE);
  constexpr int CBITS = content_bits(MODE);
  constexpr int GBYTES = group_code_bytes(CBITS);
  constexpr int ROPE_OFF = 8 * GBYTES;

  if (tid == 0) {
    for (int s = 0; s < kS; ++s) mbar_init(&sm.full[s], 1);
    for (int s = 0; s < kAggBufs; ++s) mbar_init(&sm.agg_done[s], kWarps);
    fence_mbar_init();
    fence_proxy_async();
  }
  if (w == 0) {
    tmem_alloc(&sm.tmem_base, tmem_cols<NH>());
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  int agg_ctr = 0;    // aggregation steps issued by this CTA
  int page_ctr = -1;  // the last of them that was a page step (reads every A column)
  // aggregation MMA: fp16 V^T and P^T; bf16 for an all-BF16 cache (whose
  // steps never mix with packed ones)
  constexpr uint32_t kAggIdesc = MODE == MLAQ_BF16 ? umma_idesc_bf16(128, NH) : umma_idesc_f16(128, NH);
  ProdCursor pc;
  if (tid == 0) {
    producer_init<MODE>(p, pc, first, i0, i1);
    for (int s = 0; s < kS; ++s) producer_advance<MODE>(p, sm, pc, i1);
  }

  // query fragments of heads h0 .. h0 + 15 (those of heads h0 + 16 .. h0 + 31
  // live in shared memory, one row of words per thread)
  uint32_t qf[2][4][2][2], qr[2][2], kmn[2];
  int cur_b = -1;
  const int hh = 4 * w + (lane >> 3);  // reducer lanes: head hh, tokens tp, tp+1
  const int tp = 2 * (lane & 7);
  int g = 0;                           // stages consumed by this CTA
  bool failed = false;
  int g_fail = 0;

  // Query fragments (B operand of the score MMA: k = channel, n = head) of
  // heads h0 + hoff .. h0 + hoff + 15, with the per-group query sums of the
  // min-term MMA.
  // A query element beyond +-65504 (or NaN), or a per-group query sum whose
  // fp16 split overflows, sets MLAQ_DEV_RANGE (the sequence's output is then
  // undefined; the other sequences are unaffected).
  auto make_q_frags = [&](int b, int hoff, uint32_t (&QF)[2][4][2][2], uint32_t (&QR)[2][2], uint32_t (&KM)[2]) {
    float k2[3][2];
    const uint16_t* ql = p.q_latent + ((size_t)b * H + h0) * kDL;
    const uint16_t* qp = p.q_rope + ((size_t)b * H + h0) * kDR;
    bool qbad = false;
    auto ld_q = [&](const uint16_t* src) {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(src);
      qbad |= (u & 0x7fffu) > 0x477fu || ((u >> 16) & 0x7fffu) > 0x477fu;
      if constexpr (MODE == MLAQ_BF16)
        return u;  // all-BF16 cache: bf16 score MMAs on the query as given
      else
        return bf2_to_h2(u);
    };
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int h = hoff + 8 * hb + r;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float acc = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int c = 64 * (2 * w + j) + 16 * kk + 2 * i;
          QF[j][kk][hb][0] = ld_q(ql + (size_t)h * kDL + c);
          QF[j][kk][hb][1] = ld_q(ql + (size_t)h * kDL + c + 8);
          if constexpr (MODE != MLAQ_BF16) {
            const float2 a = __half22float2(u32_as_h2(QF[j][kk][hb][0]));
            const float2 bq = __half22float2(u32_as_h2(QF[j][kk][hb][1]));
            acc += (a.x + a.y) + (bq.x + bq.y);
          }
        }
        k2[j][hb] = acc;
      }
      const int c = 16 * w + 2 * i;
      QR[hb][0] = ld_q(qp + (size_t)h * kDR + c);
      QR[hb][1] = ld_q(qp + (size_t)h * kDR + c + 8);
      if constexpr (MODE != MLAQ_BF16) {
        const float2 a = __half22float2(u32_as_h2(QR[hb][0]));
        const float2 bq = __half22float2(u32_as_h2(QR[hb][1]));
        k2[2][hb] = (a.x + a.y) + (bq.x + bq.y);
      } else {
        k2[2][hb] = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 3; ++j)
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        float v = k2[j][hb];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        k2[j][hb] = v;
      }
    // B fragment of the min-term MMA: rows k = 2j, 2j+1 hold hi/lo of K2_j
    // (an all-BF16 cache has no min term).
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      if constexpr (MODE != MLAQ_BF16) {
        const float v = (i == 0) ? k2[0][hb] : (i == 1) ? k2[1][hb] : k2[2][hb];
        qbad |= !(fabsf(v) < 65520.f);
        const __half hi = __float2half_rn(v);
        const __half lo = __float2half_rn(v - __half2float(hi));
        KM[hb] = (i < 3) ? h2_as_u32(__halves2half2(hi, lo)) : 0u;
      } else {
        KM[hb] = 0u;
      }
    }
    if (__any_sync(0xffffffffu, qbad) && lane == 0) atomicOr(p.status, MLAQ_DEV_RANGE);
  };
  // The second half's fragments: 38 words per thread, as 10 uint4 rows
  // [row][thread] (each thread reads back only its own words).
  auto store_q_frags = [&](const uint32_t (&QF)[2][4][2][2], const uint32_t (&QR)[2][2], const uint32_t (&KM)[2]) {
    if constexpr (NP == 2) {
      uint32_t wv[40];
      const uint32_t* f = &QF[0][0][0][0];
#pragma unroll
      for (int k = 0; k < 32; ++k) wv[k] = f[k];
      wv[32] = QR[0][0];
      wv[33] = QR[0][1];
      wv[34] = QR[1][0];
      wv[35] = QR[1][1];
      wv[36] = KM[0];
      wv[37] = KM[1];
      wv[38] = wv[39] = 0u;
#pragma unroll
      for (int k = 0; k < 10; ++k)
        sm.qx[k * kThreads + tid] = make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
    }
  };
  auto load_q_frags = [&](uint32_t (&QF)[2][4][2][2], uint32_t (&QR)[2][2], uint32_t (&KM)[2]) {
    if constexpr (NP == 2) {
      uint32_t wv[40];
#pragma unroll
      for (int k = 0; k < 10; ++k) {
        const uint4 v = sm.qx[k * kThreads + tid];
        wv[4 * k] = v.x;
        wv[4 * k + 1] = v.y;
        wv[4 * k + 2] = v.z;
        wv[4 * k + 3] = v.w;
      }
      uint32_t* f = &QF[0][0][0][0];
#pragma unroll
      for (int k = 0; k < 32; ++k) f[k] = wv[k];
      QR[0][0] = wv[32];
      QR[0][1] = wv[33];
      QR[1][0] = wv[34];
      QR[1][1] = wv[35];
      KM[0] = wv[36];
      KM[1] = wv[37];
    }
  };

  // Lazy-max rescale of O^T: the columns of head h times alpha[h], on this
  // warp's 32 lanes of every block (no aggregation MMA may be in flight).
  auto rescale_o = [&]() {
    float al[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) al[h] = sm.alpha[h];
#pragma unroll
    for (int blk = 0; blk < 4; ++blk)
#pragma unroll
      for (int hp = 0; hp < NP; ++hp) {
        uint32_t v[16];
        const uint32_t ta = tmem + ((uint32_t)(32 * w) << 16) + (uint32_t)(NH * blk + 16 * hp);
        tmem_ld_32x32b_x16(ta, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h) v[h] = __float_as_uint(__uint_as_float(v[h]) * al[16 * hp + h]);
        tmem_st_32x32b_x16(ta, v);
      }
    tmem_wait_st();
  };
  // Partial scores of this warp's channels (content groups 2w, 2w+1 and RoPE
  // channels 16w .. 16w+15) for 16 tokens (rows r, r + 8 of the fragments)
  // and heads hoff .. hoff + 15, published to sp[w][head][tcol + token].
  auto score_pass = [&](const uint32_t (&mx)[3], const uint32_t (&my)[3], const uint32_t (&ch)[2][4][4],
                        const uint32_t (&rf)[4], const uint32_t (&QF)[2][4][2][2], const uint32_t (&QR)[2][2],
                        const uint32_t (&KM)[2], int hoff, int tcol) {
    float sacc[2][4];  // S[t][h] for the two 8-head tiles
#pragma unroll
    for (int hb = 0; hb < 2; ++hb)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[hb][e] = 0.f;
    // min term: S += [mn_j (hi, lo) rows] . [K2_j hi, lo]
    {
      uint32_t a[4];
      const uint32_t mnx = (i == 0) ? mx[0] : (i == 1) ? mx[1] : mx[2];
      const uint32_t mny = (i == 0) ? my[0] : (i == 1) ? my[1] : my[2];
      a[0] = (i < 3) ? __byte_perm(mnx, 0, 0x3232) : 0u;  // (mn, mn)
      a[1] = (i < 3) ? __byte_perm(mny, 0, 0x3232) : 0u;
      a[2] = 0u;
      a[3] = 0u;
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) mma16816(sacc[hb], a, KM[hb], 0u);
    }
    // scale terms: D_j = codes_j . Q_j per group; the two content-group
    // chains are interleaved.
    {
      float d0[2][4], d1[2][4], d2[2][4];
#pragma unroll
      for (int hb = 0; hb < 2; ++hb)
#pragma unroll
        for (int e = 0; e < 4; ++e) d0[hb][e] = d1[hb][e] = d2[hb][e] = 0.f;
      // the RoPE term first: its segment is unpacked before the content
      // (onedev.kr "어떻게 쓰나": RoPE QK scheduled early)
      mma16816(d2[0], rf, QR[0][0], QR[0][1]);
      mma16816(d2[1], rf, QR[1][0], QR[1][1]);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma16816(d0[0], ch[0][kk], QF[0][kk][0][0], QF[0][kk][0][1]);
        mma16816(d1[0], ch[1][kk], QF[1][kk][0][0], QF[1][kk][0][1]);
        mma16816(d0[1], ch[0][kk], QF[0][kk][1][0], QF[0][kk][1][1]);
        mma16816(d1[1], ch[1][kk], QF[1][kk][1][0], QF[1][kk][1][1]);
      }
      float sxv[3], syv[3];
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        sxv[j] = __half2float(__ushort_as_half((unsigned short)(mx[j] & 0xffffu)));
        syv[j] = __half2float(__ushort_as_half((unsigned short)(my[j] & 0xffffu)));
      }
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        sacc[hb][0] = fmaf(sxv[2], d2[hb][0], fmaf(sxv[1], d1[hb][0], fmaf(sxv[0], d0[hb][0], sacc[hb][0])));
        sacc[hb][1] = fmaf(sxv[2], d2[hb][1], fmaf(sxv[1], d1[hb][1], fmaf(sxv[0], d0[hb][1], sacc[hb][1])));
        sacc[hb][2] = fmaf(syv[2], d2[hb][2], fmaf(syv[1], d1[hb][2], fmaf(syv[0], d0[hb][2], sacc[hb][2])));
        sacc[hb][3] = fmaf(syv[2], d2[hb][3], fmaf(syv[1], d1[hb][3], fmaf(syv[0], d0[hb][3], sacc[hb][3])));
      }
    }
    // publish partial scores: sacc[hb] = S[t = r (e 0,1) / r+8 (e 2,3)][h = 8hb + 2i (+1)]
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int h = hoff + 8 * hb + 2 * i;
      const int t = tcol + r;
      sm.sp[w][h][t] = sacc[hb][0];
      sm.sp[w][h + 1][t] = sacc[hb][1];
      sm.sp[w][h][t + 8] = sacc[hb][2];
      sm.sp[w][h + 1][t + 8] = sacc[hb][3];
    }
  };

  // The score pass of an all-BF16 cache: (s, mn) = (1, 0), so the partial
  // score is one chain of bf16 MMAs over the warp's 144 channels.
  auto score_pass_bf16 = [&](const uint32_t (&ch)[2][4][4], const uint32_t (&rf)[4],
                             const uint32_t (&QF)[2][4][2][2], const uint32_t (&QR)[2][2], int hoff) {
    float sacc[2][4];
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[hb][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma16816_bf16(sacc[hb], ch[0][kk], QF[0][kk][hb][0], QF[0][kk][hb][1]);
        mma16816_bf16(sacc[hb], ch[1][kk], QF[1][kk][hb][0], QF[1][kk][hb][1]);
      }
      mma16816_bf16(sacc[hb], rf, QR[hb][0], QR[hb][1]);
    }
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int h = hoff + 8 * hb + 2 * i;
      sm.sp[w][h][r] = sacc[hb][0];
      sm.sp[w][h + 1][r] = sacc[hb][1];
      sm.sp[w][h][r + 8] = sacc[hb][2];
      sm.sp[w][h + 1][r + 8] = sacc[hb][3];
    }
  };

  for (int item_idx = i0; item_idx < i1; ++item_idx) {
    const Item it = p.items[item_idx];
    const int L = it.L;
    const bool single = p.item_start[it.b + 1] - p.item_start[it.b] == 1;
    if (it.b != cur_b) {
      cur_b = it.b;
      make_q_frags(it.b, 0, qf, qr, kmn);
      if constexpr (NP == 2) {
        uint32_t q1f[2][4][2][2], q1r[2][2], q1k[2];
        make_q_frags(it.b, 16, q1f, q1r, q1k);
        store_q_frags(q1f, q1r, q1k);
      }
    }

    bool item_first = true;  // the item's first aggregation MMA overwrites O^T
    float m_run[NP], l_run[NP];  // per 16-head half: heads hh (+ 16)
#pragma unroll
    for (int hp = 0; hp < NP; ++hp) {
      m_run[hp] = -INFINITY;
      l_run[hp] = 0.f;
    }

    const int nst = item_stages<MODE>(it, L);
    for (int k = 0; k < nst && !failed; ++k) {
      const int buf = g % kS;
      const bool ok = mbar_wait_bounded(&sm.full[buf], (g / kS) & 1, kWaitLimit);
      g++;
      const uint8_t* st = sm.stage[buf];
      const bool bad = sm.stage_bad[buf] != 0;
      const StageRef sref = item_stage<MODE>(it, L, k);
      const bool packed = sref.kind == 1;
      const int nsteps = packed ? kPage / kT : 1;
      // One 16-token step. FULL: a packed step of a live stage whose 16 rows
      // are all valid (inside [4, L - 128)), the common case, compiled
      // without any per-row masking.
      auto step_body = [&](auto full_c, const int s) -> bool {
        constexpr bool FULL = decltype(full_c)::value;
        const bool packed_s = FULL || packed;
        const int lr = s * kT + r;  // row of token r in the stage
        bool all_in = FULL;         // every row of the step valid
        if (!FULL && packed) {
          const int t0 = kPage * sref.idx + s * kT;
          all_in = t0 >= kSink && t0 + kT <= L - kRecent;
        }
        const bool live = FULL || (ok & !bad);
        const bool v0 = FULL || (live & (all_in | row_valid<MODE>(sref, lr, L)));
        const bool v1 = FULL || (live & (all_in | row_valid<MODE>(sref, lr + 8, L)));
        // ---------------- dequant + scores
        uint32_t mx[3], my[3];  // meta (s, mn) of tokens r (x) and r+8 (y), groups 2w, 2w+1, rope
        uint32_t ch[2][4][4];   // fp16 A fragments of the content tile (exact codes, later dequantized)
        uint32_t rf[4];
        if (packed_s) {
          const uint8_t* mtab = st + page_code_bytes(MODE);
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const int gg = j < 2 ? 2 * w + j : 8;
            const uint32_t mxr = *reinterpret_cast<const uint32_t*>(mtab + lr * kMetaTok + 4 * gg);
            const uint32_t myr = *reinterpret_cast<const uint32_t*>(mtab + (lr + 8) * kMetaTok + 4 * gg);
            mx[j] = v0 ? mxr : 0u;
            my[j] = v1 ? myr : 0u;
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int gg = 2 * w + j;
            if constexpr (CBITS == 4) {
              const uint2 wx = *reinterpret_cast<const uint2*>(st + lr * CB + gg * GBYTES + 8 * i);
              const uint2 wy = *reinterpret_cast<const uint2*>(st + (lr + 8) * CB + gg * GBYTES + 8 * i);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t ax = (kk >> 1) ? wx.y : wx.x, ay = (kk >> 1) ? wy.y : wy.x;
                const uint32_t ax8 = ax >> 8, ay8 = ay >> 8;
                const int p0 = 2 * (kk & 1);
                ch[j][kk][0] = int4_pos(ax, ax8, p0);
                ch[j][kk][1] = int4_pos(ay, ay8, p0);
                ch[j][kk][2] = int4_pos(ax, ax8, p0 + 1);
                ch[j][kk][3] = int4_pos(ay, ay8, p0 + 1);
              }
            } else {
              const uint32_t ax = *reinterpret_cast<const uint32_t*>(st + lr * CB + gg * GBYTES + 4 * i);
              const uint32_t ay = *reinterpret_cast<const uint32_t*>(st + (lr + 8) * CB + gg * GBYTES + 4 * i);
              const uint32_t ax8 = ax >> 8, ay8 = ay >> 8;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                ch[j][kk][0] = int2_pos(ax, ax8, 2 * kk);
                ch[j][kk][1] = int2_pos(ay, ay8, 2 * kk);
                ch[j][kk][2] = int2_pos(ax, ax8, 2 * kk + 1);
                ch[j][kk][3] = int2_pos(ay, ay8, 2 * kk + 1);
              }
            }
          }
          {
            uint32_t ax = *reinterpret_cast<const uint32_t*>(st + lr * CB + ROPE_OFF + 4 * (2 * w + (i >> 1)));
            uint32_t ay = *reinterpret_cast<const uint32_t*>(st + (lr + 8) * CB + ROPE_OFF + 4 * (2 * w + (i >> 1)));
            if (i & 1) {
              ax >>= 8;
              ay >>= 8;
            }
            rf[0] = int4_pos(ax, 0u, 0);
            rf[1] = int4_pos(ay, 0u, 0);
            rf[2] = int4_pos(ax, 0u, 1);
            rf[3] = int4_pos(ay, 0u, 1);
          }
        } else {
          // BF16 tokens (ring or all-BF16 pages): q = x, (s, mn) = (1, 0)
          const uint32_t one = 0x00003C00u;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            mx[j] = v0 ? one : 0u;
            my[j] = v1 ? one : 0u;
          }
          // One ldmatrix.x4 per 16 x 16 fragment: lane L gives the address of
          // row 8 (L / 8 % 2) + L % 8 of the step at the 16-byte chunk q + L / 16
          // (channels 8q .. 8q + 7, q = (16-channel block) / 8); rows keep their
          // chunks XOR-permuted by the row index mod 8, so each 8 x 8 matrix
          // reads eight distinct bank groups. The registers come back in the
          // A-fragment order: rows r / r + 8, channels 2i, 2i + 1 (+ 8).
          const int mrow = s * kT + 8 * ((lane >> 3) & 1) + (lane & 7);
          const uint32_t rowa = smem_u32(st + mrow * (kD * 2));
          auto frag = [&](int q, uint32_t (&f)[4]) {
            ldmatrix_x4(rowa + ((uint32_t)((q + (lane >> 4)) ^ (lane & 7)) << 4), f);
            f[0] = v0 ? bf_operand<MODE>(f[0]) : 0u;
            f[1] = v1 ? bf_operand<MODE>(f[1]) : 0u;
            f[2] = v0 ? bf_operand<MODE>(f[2]) : 0u;
            f[3] = v1 ? bf_operand<MODE>(f[3]) : 0u;
          };
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) frag(8 * (2 * w + j) + 2 * kk, ch[j][kk]);
          frag(kDL / 8 + 2 * w, rf);
        }
        if constexpr (MODE == MLAQ_BF16) {
          score_pass_bf16(ch, rf, qf, qr, 0);
          if constexpr (NP == 2) {
            uint32_t q1f[2][4][2][2], q1r[2][2], q1k[2];
            load_q_frags(q1f, q1r, q1k);
            score_pass_bf16(ch, rf, q1f, q1r, 16);
          }
        } else {
          score_pass(mx, my, ch, rf, qf, qr, kmn, 0, 0);
          if constexpr (NP == 2) {
            uint32_t q1f[2][4][2][2], q1r[2][2], q1k[2];
            load_q_frags(q1f, q1r, q1k);
            score_pass(mx, my, ch, rf, q1f, q1r, q1k, 16, 0);
          }
        }
        // dequantize the content tile in place (fp16, one rounding; bf16
        // tokens of an all-BF16 cache are the values themselves) and
        // transpose each 8x8 block for the aggregation B operand.
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const __half2 s2x = __low2half2(u32_as_h2(mx[j])), m2x = __high2half2(u32_as_h2(mx[j]));
          const __half2 s2y = __low2half2(u32_as_h2(my[j])), m2y = __high2half2(u32_as_h2(my[j]));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if constexpr (MODE == MLAQ_BF16) {
#pragma unroll
              for (int e = 0; e < 4; ++e) ch[j][kk][e] = movmatrix_t(ch[j][kk][e]);
            } else {
              ch[j][kk][0] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][0]), s2x, m2x)));
              ch[j][kk][1] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][1]), s2y, m2y)));
              ch[j][kk][2] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][2]), s2x, m2x)));
              ch[j][kk][3] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][3]), s2y, m2y)));
            }
          }
        }
        // content tile -> TMEM A step buffer (lanes = channels, columns = token pairs)
        const int ab = agg_ctr % kAggBufs;
        bool agg_ok = true;
        {
          // the MMAs that last read buffer ab (two steps back), or a later
          // page step's, which read every A column, must be complete
          const int lp = max(agg_ctr - kAggBufs, page_ctr);
          if (lp >= 0) agg_ok = mbar_wait_bounded(&sm.agg_done[lp % kAggBufs], (lp / kAggBufs) & 1, kWaitLimit);
        }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int blk = 2 * j + (kk >> 1);
            const uint32_t ta = tmem + ((uint32_t)(32 * w + 16 * (kk & 1)) << 16) +
                                (uint32_t)(kTmemA + 32 * ab + 8 * blk);
            tmem_st_16x256b(ta, ch[j][kk][0], ch[j][kk][1], ch[j][kk][2], ch[j][kk][3]);
          }
        tmem_wait_st();
        tc_fence_before();
        // barrier 1: partial scores complete; also agrees on a timed-out wait
        if (named_bar_or(1, kThreads, !(ok && agg_ok))) return true;
        // the stage's shared memory is no longer read: refill it with the
        // next stage of the CTA's stream
        if (tid == 0 && s == nsteps - 1) producer_advance<MODE>(p, sm, pc, i1);
        // ---------------- online softmax for heads hh (+ 16), tokens tp, tp+1
        {
          const bool ok0 = FULL || (!bad & (all_in | row_valid<MODE>(sref, s * kT + tp, L)));
          const bool ok1 = FULL || (!bad & (all_in | row_valid<MODE>(sref, s * kT + tp + 1, L)));
          const int kp = tp < 8 ? 2 * tp : 2 * tp - 14;  // P^T token order matching the TMEM A columns
          bool rs = false;
#pragma unroll
          for (int hp = 0; hp < NP; ++hp) {
            const int hq = hh + 16 * hp;
            bool ok0h = ok0, ok1h = ok1;
            if (p.q_len > 1) {  // query j of several sees t < L - (q_len - 1 - j)
              const int lim = L - (p.q_len - 1 - (h0 + hq) / p.h_per_q);
              ok0h = ok0h && row_token<MODE>(sref, s * kT + tp, L) < lim;
              ok1h = ok1h && row_token<MODE>(sref, s * kT + tp + 1, L) < lim;
            }
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) {
              const float2 v = *reinterpret_cast<const float2*>(&sm.sp[ww][hq][tp]);
              x0 += v.x;
              x1 += v.y;
            }
            x0 = ok0h ? x0 * p.scale_log2 : -INFINITY;
            x1 = ok1h ? x1 * p.scale_log2 : -INFINITY;
            // Lazy rescale: keep a stale running max while every P <= 2^14 (fp16
            // holds it exactly enough; the sums are fp32). The tile max (three
            // shuffles) is only needed when some score exceeds it by more than
            // 14 (log2 units), e.g. on an item's first tile.
            float alpha = 1.f;
            if (__any_sync(0xffffffffu, fmaxf(x0, x1) > m_run[hp] + 14.f)) {
              float tmax = fmaxf(x0, x1);
              tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
              tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
              tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
              const bool upd = tmax > m_run[hp] + 14.f;  // m_run = -inf gives alpha = 0
              alpha = upd ? ex2(m_run[hp] - tmax) : 1.f;
              m_run[hp] = upd ? tmax : m_run[hp];
            }
            const float mref = (m_run[hp] == -INFINITY) ? 0.f : m_run[hp];  // nothing valid yet: p = 0
            const float p0 = ex2(x0 - mref), p1 = ex2(x1 - mref);
            l_run[hp] = l_run[hp] * alpha + (p0 + p1);
            const int off = (hq >> 3) * 256 + (kp >> 3) * 128 + (hq & 7) * 16 + (kp & 7) * 2;
            if constexpr (MODE == MLAQ_BF16)
              *reinterpret_cast<__nv_bfloat162*>(&sm.pt[ab][off]) = __floats2bfloat162_rn(p0, p1);
            else
              *reinterpret_cast<__half2*>(&sm.pt[ab][off]) = __floats2half2_rn(p0, p1);
            if ((lane & 7) == 0) sm.alpha[hq] = alpha;
            rs |= alpha != 1.f;
          }
          fence_view_async_shared();
          const bool any_rs = __any_sync(0xffffffffu, rs);
          if (lane == 0) sm.rescale_flag[w] = any_rs;
        }
        named_bar_sync(2, kThreads);
        // ---------------- aggregation
        {
          const bool need_rs = !item_first && (sm.rescale_flag[0] | sm.rescale_flag[1] | sm.rescale_flag[2] |
                                               sm.rescale_flag[3]);
          if (need_rs) {  // rare (lazy max): scale O^T columns by alpha[head]
            const int lp = agg_ctr - 1;
            mbar_wait_bounded(&sm.agg_done[lp % kAggBufs], (lp / kAggBufs) & 1, kWaitLimit);
            tc_fence_after();
            rescale_o();
            tc_fence_before();
            named_bar_sync(3, kThreads);
            tc_fence_after();
          }
          if (lane == 0) {
            tc_fence_after();
            const uint64_t bdesc = umma_smem_desc(smem_u32(sm.pt[ab]), 128, 256);
            umma_f16_ts(tmem + (uint32_t)(NH * w), tmem + (uint32_t)(kTmemA + 32 * ab + 8 * w), bdesc, kAggIdesc,
                        !item_first);
            umma_commit(&sm.agg_done[ab]);
          }
          __syncwarp();
          item_first = false;
          agg_ctr++;
        }
        // No barrier before the next step's writes to sp: every thread passed
        // barrier 2 after all reads of sp; pr/alpha are rewritten only after
        // the next barrier 1, which all threads reach after their reads.
        return false;
      };
      // A whole packed page (64 tokens, all valid) under one pair of
      // barriers. The four 16-token sub-steps store their dequantized,
      // transposed content tiles in TMEM (A operand, lanes = channels) and
      // publish partial scores; after the softmax of all 64 tokens each warp
      // issues four tcgen05 MMAs (its 128-channel block) that accumulate
      // O^T += V^T P^T asynchronously.
      // MASKED: rows outside the packed range [4, L - 128) contribute nothing
      // (zero scale and min, score -inf); the first and last pages of a range.
      auto page_body = [&](auto masked_c, const int part) -> bool {
        constexpr bool MASKED = decltype(masked_c)::value;
        bool agg_ok = true;
        if (agg_ctr > 0) {  // every earlier aggregation MMA has read its TMEM/smem operands
          const int lp = agg_ctr - 1;
          agg_ok = mbar_wait_bounded(&sm.agg_done[lp % kAggBufs], (lp / kAggBufs) & 1, kWaitLimit);
        }
        tc_fence_after();
        const uint8_t* mtab = st + page_code_bytes(MODE);
#pragma unroll 1
        for (int sub = 0; sub < kSubs; ++sub) {
          const int lr = 16 * (kSubs * part + sub) + r;
          bool v0 = true, v1 = true;
          if constexpr (MASKED) {
            const int t = kPage * sref.idx + lr;
            v0 = (t >= kSink) & (t < L - kRecent);
            v1 = (t + 8 >= kSink) & (t + 8 < L - kRecent);
          }
          uint32_t mx[3], my[3];
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const int gg = j < 2 ? 2 * w + j : 8;
            const uint32_t mxr = *reinterpret_cast<const uint32_t*>(mtab + lr * kMetaTok + 4 * gg);
            const uint32_t myr = *reinterpret_cast<const uint32_t*>(mtab + (lr + 8) * kMetaTok + 4 * gg);
            mx[j] = v0 ? mxr : 0u;
            my[j] = v1 ? myr : 0u;
          }
          uint32_t rf[4];  // the RoPE slice first (its MMAs lead the score pass)
          {
            uint32_t ax = *reinterpret_cast<const uint32_t*>(st + lr * CB + ROPE_OFF + 4 * (2 * w + (i >> 1)));
            uint32_t ay = *reinterpret_cast<const uint32_t*>(st + (lr + 8) * CB + ROPE_OFF + 4 * (2 * w + (i >> 1)));
            if (i & 1) {
              ax >>= 8;
              ay >>= 8;
            }
            rf[0] = int4_pos(ax, 0u, 0);
            rf[1] = int4_pos(ay, 0u, 0);
            rf[2] = int4_pos(ax, 0u, 1);
            rf[3] = int4_pos(ay, 0u, 1);
          }
          uint32_t ch[2][4][4];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int gg = 2 * w + j;
            if constexpr (CBITS == 4) {
              const uint2 wx = *reinterpret_cast<const uint2*>(st + lr * CB + gg * GBYTES + 8 * i);
              const uint2 wy = *reinterpret_cast<const uint2*>(st + (lr + 8) * CB + gg * GBYTES + 8 * i);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t ax = (kk >> 1) ? wx.y : wx.x, ay = (kk >> 1) ? wy.y : wy.x;
                const uint32_t ax8 = ax >> 8, ay8 = ay >> 8;
                const int p0 = 2 * (kk & 1);
                ch[j][kk][0] = int4_pos(ax, ax8, p0);
                ch[j][kk][1] = int4_pos(ay, ay8, p0);
                ch[j][kk][2] = int4_pos(ax, ax8, p0 + 1);
                ch[j][kk][3] = int4_pos(ay, ay8, p0 + 1);
              }
            } else {
              const uint32_t ax = *reinterpret_cast<const uint32_t*>(st + lr * CB + gg * GBYTES + 4 * i);
              const uint32_t ay = *reinterpret_cast<const uint32_t*>(st + (lr + 8) * CB + gg * GBYTES + 4 * i);
              const uint32_t ax8 = ax >> 8, ay8 = ay >> 8;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                ch[j][kk][0] = int2_pos(ax, ax8, 2 * kk);
                ch[j][kk][1] = int2_pos(ay, ay8, 2 * kk);
                ch[j][kk][2] = int2_pos(ax, ax8, 2 * kk + 1);
                ch[j][kk][3] = int2_pos(ay, ay8, 2 * kk + 1);
              }
            }
          }
          score_pass(mx, my, ch, rf, qf, qr, kmn, 0, 16 * sub);
          if constexpr (NP == 2) {
            uint32_t q1f[2][4][2][2], q1r[2][2], q1k[2];
            load_q_frags(q1f, q1r, q1k);
            score_pass(mx, my, ch, rf, q1f, q1r, q1k, 16, 16 * sub);
          }
          // dequantize, transpose, and store the sub-step's A tile in TMEM
          // (lanes = channels, columns = token pairs)
          uint32_t vv[2][16];  // [kk & 1][column block blk = 2j + kk / 2][4 registers]
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const __half2 s2x = __low2half2(u32_as_h2(mx[j])), m2x = __high2half2(u32_as_h2(mx[j]));
            const __half2 s2y = __low2half2(u32_as_h2(my[j])), m2y = __high2half2(u32_as_h2(my[j]));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const int blk = 2 * j + (kk >> 1);
              uint32_t* v = &vv[kk & 1][4 * blk];
              v[0] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][0]), s2x, m2x)));
              v[1] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][1]), s2y, m2y)));
              v[2] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][2]), s2x, m2x)));
              v[3] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][3]), s2y, m2y)));
            }
          }
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2)
            tmem_st_16x256b_x4(tmem + ((uint32_t)(32 * w + 16 * k2) << 16) + (uint32_t)(kTmemA + 32 * sub), vv[k2]);
        }
        tmem_wait_st();
        tc_fence_before();
        // barrier 1: partial scores and A tiles complete; agrees on a timed-out wait
        if (named_bar_or(1, kThreads, !(ok && agg_ok))) return true;
        if (tid == 0 && part == kPageParts - 1) producer_advance<MODE>(p, sm, pc, i1);
        // online softmax for heads hh (+ 16), tokens tq .. tq + 3 (and 32 + tq .. 32 + tq + 3
        // in whole pages) of the body (a quarter warp reads 128 contiguous bytes of a score row)
        {
          constexpr int NU = 2 * kSubs;  // tokens per thread
          const int tq = 4 * (lane & 7);
          bool rs = false;
#pragma unroll
          for (int hp = 0; hp < NP; ++hp) {
            const int hq = hh + 16 * hp;
            float x[NU];
#pragma unroll
            for (int u = 0; u < NU; ++u) x[u] = 0.f;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) {
#pragma unroll
              for (int u4 = 0; u4 < NU; u4 += 4) {
                const float4 v = *reinterpret_cast<const float4*>(&sm.sp[ww][hq][tq + 8 * u4]);
                x[u4] += v.x;
                x[u4 + 1] += v.y;
                x[u4 + 2] += v.z;
                x[u4 + 3] += v.w;
              }
            }
            float xm = -INFINITY;
#pragma unroll
            for (int u = 0; u < NU; ++u) {
              bool valid = true;
              if constexpr (MASKED) {
                const int t = kPage * sref.idx + 16 * kSubs * part + tq + (u < 4 ? u : 28 + u);
                valid = (t >= kSink) & (t < L - kRecent);
              }
              x[u] = valid ? x[u] * p.scale_log2 : -INFINITY;
              xm = fmaxf(xm, x[u]);
            }
            float alpha = 1.f;
            if (__any_sync(0xffffffffu, xm > m_run[hp] + 14.f)) {
              float tmax = xm;
              tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
              tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
              tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
              const bool upd = tmax > m_run[hp] + 14.f;
              alpha = upd ? ex2(m_run[hp] - tmax) : 1.f;
              m_run[hp] = upd ? tmax : m_run[hp];
            }
            float psum = 0.f;
            const float mref = (MASKED && m_run[hp] == -INFINITY) ? 0.f : m_run[hp];  // nothing valid yet: p = 0
#pragma unroll
            for (int u = 0; u < NU; u += 2) {
              const float pa = ex2(x[u] - mref), pb = ex2(x[u + 1] - mref);
              psum += pa + pb;
              const int tp64 = tq + (u < 4 ? u : 28 + u);  // token pair tp64, tp64 + 1 of the body
              const int sub = tp64 >> 4, t = tp64 & 15;
              const int kp = t < 8 ? 2 * t : 2 * t - 14;  // their K index in the TMEM A columns
              const int off = (hq >> 3) * 256 + (kp >> 3) * 128 + (hq & 7) * 16 + (kp & 7) * 2;
              *reinterpret_cast<__half2*>(&sm.ptp[sub][off]) = __floats2half2_rn(pa, pb);
            }
            l_run[hp] = l_run[hp] * alpha + psum;
            if ((lane & 7) == 0) sm.alpha[hq] = alpha;
            rs |= alpha != 1.f;
          }
          fence_view_async_shared();
          const bool any_rs = __any_sync(0xffffffffu, rs);
          if (lane == 0) sm.rescale_flag[w] = any_rs;
        }
        named_bar_sync(2, kThreads);
        {
          const bool need_rs = !item_first && (sm.rescale_flag[0] | sm.rescale_flag[1] | sm.rescale_flag[2] |
                                               sm.rescale_flag[3]);
          if (need_rs) {  // rare (lazy max): scale O^T columns by alpha[head]; no MMA is in flight
            rescale_o();
            tc_fence_before();
            named_bar_sync(3, kThreads);
            tc_fence_after();
          }
          if (lane == 0) {
            tc_fence_after();
#pragma unroll
            for (int sub = 0; sub < kSubs; ++sub) {
              const uint64_t bdesc = umma_smem_desc(smem_u32(sm.ptp[sub]), 128, 256);
              umma_f16_ts(tmem + (uint32_t)(NH * w), tmem + (uint32_t)(kTmemA + 32 * sub + 8 * w), bdesc,
                          kAggIdesc, !item_first || sub > 0);
            }
            umma_commit(&sm.agg_done[agg_ctr % kAggBufs]);
          }
          __syncwarp();
          item_first = false;
          page_ctr = agg_ctr;
          agg_ctr++;
        }
        return false;
      };
      if constexpr (MODE != MLAQ_BF16) {
        if (packed) {
          const int t0 = kPage * sref.idx;
          if (!bad) {  // CTA-uniform
            const bool full = t0 >= kSink && t0 + kPage <= L - kRecent;
            for (int part = 0; part < kPageParts; ++part) {
              if (full ? page_body(BoolC<false>{}, part) : page_body(BoolC<true>{}, part)) {
                failed = true;
                g_fail = g - 1;
                break;
              }
            }
            continue;
          }
        }
      }
      for (int s = 0; s < nsteps; ++s) {
        bool full = false;
        if (packed) {
          const int t0 = kPage * sref.idx + s * kT;
          full = ok & !bad & (t0 >= kSink) & (t0 + kT <= L - kRecent);
        }
        // both variants meet at the same named barriers, so threads that
        // disagree on `full` (a timed-out wait is per thread) stay in step
        bool fail;
        if constexpr (MODE == MLAQ_BF16)
          fail = step_body(BoolC<false>{}, s);  // no packed steps
        else
          fail = full ? step_body(BoolC<true>{}, s) : step_body(BoolC<false>{}, s);
        if (fail) {
          failed = true;
          g_fail = g - 1;
          break;
        }
      }
    }

    // ---- item epilogue: normalized partial O and lse for heads h0 .. h0 + NH - 1
#pragma unroll
    for (int hp = 0; hp < NP; ++hp) {
      float l_tot = l_run[hp];
      l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
      l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
      l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 4);
      if ((lane & 7) == 0) {
        sm.fin_m[hh + 16 * hp] = m_run[hp];
        sm.fin_l[hh + 16 * hp] = failed ? 0.f : l_tot;
      }
    }
    __syncthreads();
    // A sequence with a single item is final here (bf16 out, lse); otherwise
    // the normalized partial (fp16) and its lse go to the combine kernel.
    __half* op = p.o_part + ((size_t)item_idx * H + h0) * kDL;
    {
      // O^T lane l of block blk holds channel 128 (l/32) + 64 (blk/2) + 16 (2 (blk%2) + (l%32)/16) + l%16
      if (agg_ctr > 0) {
        const int lp = agg_ctr - 1;
        mbar_wait_bounded(&sm.agg_done[lp % kAggBufs], (lp / kAggBufs) & 1, kWaitLimit);
      }
      tc_fence_after();
      const int x = lane;
#pragma unroll
      for (int hp = 0; hp < NP; ++hp) {
        float inv[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float l = sm.fin_l[16 * hp + h];
          inv[h] = l > 0.f ? 1.f / l : 0.f;
        }
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + ((uint32_t)(32 * w) << 16) + (uint32_t)(NH * blk + 16 * hp), v);
          tmem_wait_ld();
          const int c = 128 * w + 64 * (blk >> 1) + 16 * (2 * (blk & 1) + (x >> 4)) + (x & 15);
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const int hq = 16 * hp + h;
            const float val = inv[h] != 0.f ? __uint_as_float(v[h]) * inv[h] : 0.f;
            if (single)
              p.out[((size_t)it.b * H + h0 + hq) * kDL + c] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
            else
              op[(size_t)hq * kDL + c] = __float2half_rn(val);
          }
        }
      }
      tc_fence_before();
    }
    if (tid < NH) {
      const float l = sm.fin_l[tid];
      const float lse_v = l > 0.f ? (sm.fin_m[tid] + log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (single)
        p.lse[(size_t)it.b * H + h0 + tid] = lse_v;
      else
        p.lse_part[(size_t)item_idx * H + h0 + tid] = lse_v;
    }
    __syncthreads();  // fin_* are reused by the next item
  }

  if (failed && tid == 0) {
    atomicOr(p.status, MLAQ_DEV_TIMEOUT);
    // wait (bounded) for copies still in flight before the CTA exits
    for (int gg = g_fail; gg < pc.issued; ++gg)
      mbar_wait_bounded(&sm.full[gg % kS], (gg / kS) & 1, kWaitLimit);
  }
  // every aggregation MMA has completed (waited for in each item epilogue)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (w == 0) tmem_dealloc(tmem, tmem_cols<NH>());
}

}  // namespace mlaq

#include "mlaq_decode_tc.cuh"

namespace mlaq {

// ---------------------------------------------------------------------------
// Combine (split-KV): for every sequence with more than one item, the
// normalized partials O_k and their lse_k merge into
//   out = sum_k exp(lse_k - M) O_k / sum_k exp(lse_k - M),  lse = M + log(sum_k exp(lse_k - M)).
// One work unit = (sequence, 16-head block, chunk of 8 CPT channels); a thread
// owns one head and CPT channels and reads BATCH partials per round trip.
// CPT = 4 with BATCH = 16 reads a sequence split up to 16 ways in one round
// trip; CPT = 16 with BATCH = 4 serves large batches with a quarter of the
// CTAs (one wave where the small units would need several).
template <int CPT, int BATCH>
__global__ void __launch_bounds__(128) combine_kernel(DecodeParams p) {
  constexpr int kChunks = kDL / (8 * CPT);
  constexpr int NV = CPT / 4;  // uint2 (4 fp16) words per partial
  const int tid = threadIdx.x;
  const int hc = tid >> 3, cq = (tid & 7) * CPT;  // head in the block, channels of the chunk
  const int HB16 = p.H / 16;
  const int units = p.B * HB16 * kChunks;
  // The item ranges come from the plan, which completed before the decode
  // grid started (and so before this grid was launched): they are read
  // before waiting for the decode grid.
  int u = blockIdx.x;
  int s0 = 0, s1 = 0;
  if (u < units) {
    const int b = (u / kChunks) / HB16;
    s0 = p.item_start[b];
    s1 = p.item_start[b + 1];
  }
  pdl_wait();
  for (; u < units; u += gridDim.x) {
    const int chunk = u % kChunks, rest = u / kChunks;
    const int hb = rest % HB16, b = rest / HB16;
    if (u != (int)blockIdx.x) {
      s0 = p.item_start[b];
      s1 = p.item_start[b + 1];
    }
    if (s1 - s0 < 2) continue;  // finalized by the decode kernel
    const int row = 16 * hb + hc;
    const int c = 8 * CPT * chunk + cq;
    // one pass over the partials, BATCH at a time, with a running max
    float m = -INFINITY, tot = 0.f;
    float acc[CPT];
#pragma unroll
    for (int e = 0; e < CPT; ++e) acc[e] = 0.f;
    for (int k0 = s0; k0 < s1; k0 += BATCH) {
      uint2 v[BATCH][NV];
      float l[BATCH];
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        const bool in = k0 + k < s1;
        l[k] = in ? __ldcg(&p.lse_part[(size_t)(k0 + k) * p.H + row]) : -INFINITY;
        const uint2* src = reinterpret_cast<const uint2*>(p.o_part + ((size_t)(k0 + k) * p.H + row) * kDL + c);
#pragma unroll
        for (int q = 0; q < NV; ++q) v[k][q] = in ? __ldcg(src + q) : make_uint2(0u, 0u);
      }
      float mb = m;
#pragma unroll
      for (int k = 0; k < BATCH; ++k) mb = fmaxf(mb, l[k]);
      if (mb == -INFINITY) continue;  // no tokens so far
      const float sc = expf(m - mb);  // 0 while m = -inf
      tot *= sc;
#pragma unroll
      for (int e = 0; e < CPT; ++e) acc[e] *= sc;
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        const float wgt = expf(l[k] - mb);  // 0 for padding (lse = -inf)
        tot += wgt;
#pragma unroll
        for (int q = 0; q < NV; ++q) {
          const __half2* hv = reinterpret_cast<const __half2*>(&v[k][q]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float2 f = __half22float2(hv[e]);
            acc[4 * q + 2 * e] = fmaf(wgt, f.x, acc[4 * q + 2 * e]);
            acc[4 * q + 2 * e + 1] = fmaf(wgt, f.y, acc[4 * q + 2 * e + 1]);
          }
        }
      }
      m = mb;
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    uint2* dst = reinterpret_cast<uint2*>(p.out + ((size_t)b * p.H + row) * kDL + c);
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      uint2 pk;
      uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const __nv_bfloat162 bv = __floats2bfloat162_rn(acc[4 * q + 2 * e] * inv, acc[4 * q + 2 * e + 1] * inv);
        pw[e] = *reinterpret_cast<const uint32_t*>(&bv);
      }
      dst[q] = pk;
    }
    if (chunk == 0 && (tid & 7) == 0) p.lse[(size_t)b * p.H + row] = tot > 0.f ? m + logf(tot) : -INFINITY;
  }
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream finishes; it calls pdl_wait() before it
// reads anything that kernel wrote.
template <typename... Args>
static cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Opt every decode-path kernel into its dynamic shared memory (> 48 KB), once
// per device and for all variants together, so that the first decode call on
// a device, whatever its mode and head count, is the only one that changes a
// function attribute (it must run outside a stream capture). Serialised
// across host threads.
template <int MODE, int NH>
static cudaError_t set_decode_attr() {
  return cudaFuncSetAttribute(decode_kernel<MODE, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(DecodeSmem<NH>));
}
template <int MODE, int NH>
static cudaError_t set_decode_tc_attr() {
  return cudaFuncSetAttribute(decode_tc_kernel<MODE, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(TcSmem<NH>));
}
static cudaError_t set_all_decode_attrs() {
  const cudaError_t es[] = {
      set_decode_attr<MLAQ_C4R4, 16>(), set_decode_attr<MLAQ_C2R4, 16>(), set_decode_attr<MLAQ_BF16, 16>(),
      set_decode_attr<MLAQ_C4R4, 32>(), set_decode_attr<MLAQ_C2R4, 32>(), set_decode_attr<MLAQ_BF16, 32>(),
      set_decode_tc_attr<MLAQ_C4R4, 16>(), set_decode_tc_attr<MLAQ_C2R4, 16>(), set_decode_tc_attr<MLAQ_BF16, 16>(),
      set_decode_tc_attr<MLAQ_C4R4, 32>(), set_decode_tc_attr<MLAQ_C2R4, 32>(), set_decode_tc_attr<MLAQ_BF16, 32>(),
      set_decode_tc_attr<MLAQ_C4R4, 64>(), set_decode_tc_attr<MLAQ_C2R4, 64>(), set_decode_tc_attr<MLAQ_BF16, 64>(),
      // the planner's shared-memory arrays exceed 48 KB for large batches
      cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)plan_smem_bytes(kMaxSeqs, kMaxPlanCtas))};
  for (cudaError_t e : es)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}
static std::mutex g_attr_mutex;
static std::atomic<bool> g_attr_done[kMaxDevices];
cudaError_t decode_attrs_ready() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return set_all_decode_attrs();
  if (g_attr_done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  if (g_attr_done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = set_all_decode_attrs();
  if (e == cudaSuccess) g_attr_done[dev].store(true, std::memory_order_release);
  return e;
}

// The combine after the attention kernel, and the call's closing event.
static cudaError_t launch_combine(mlaq_cache* c, const DecodeParams& p, cudaStream_t s, cudaError_t e,
                                  cudaEvent_t* ev) {
  if (e == cudaSuccess) {
    // one unit per CTA, every unit's partial loads in one round trip; large
    // batches take the 16-channel units so that the grid stays near one wave
    const int small_units = p.B * (p.H / 16) * (kDL / 32);
    if (small_units <= 16 * max(1, c->num_sms))
      e = launch_pdl(combine_kernel<4, 16>, dim3(max(1, small_units)), dim3(128), 0, s, p);
    else
      e = launch_pdl(combine_kernel<16, 4>, dim3(max(1, small_units / 4)), dim3(128), 0, s, p);
  }
  if (ev) {
    cudaEventRecord(ev[1], s);
    c->timing_n++;
  }
  return e;
}

template <int MODE, int NH>
static cudaError_t run_decode_tc(mlaq_cache* c, const DecodeParams& p, int grid_cta, cudaStream_t s) {
  cudaEvent_t* ev = nullptr;
  if (c->timing_events && c->timing_n < c->timing_max)
    ev = reinterpret_cast<cudaEvent_t*>(c->timing_events) + 2 * c->timing_n;  // ev[0] precedes the plan
  const cudaError_t e = launch_pdl(decode_tc_kernel<MODE, NH>, dim3(p.HB, grid_cta), dim3(TcCfg<NH>::kThreads),
                                   sizeof(TcSmem<NH>), s, p);
  return launch_combine(c, p, s, e, ev);
}

template <int MODE, int NH>
static cudaError_t run_decode(mlaq_cache* c, const DecodeParams& p, int grid_cta, cudaStream_t s) {
  const int smem = (int)sizeof(DecodeSmem<NH>);
  cudaEvent_t* ev = nullptr;
  if (c->timing_events && c->timing_n < c->timing_max)
    ev = reinterpret_cast<cudaEvent_t*>(c->timing_events) + 2 * c->timing_n;  // ev[0] precedes the plan
  const cudaError_t e = launch_pdl(decode_kernel<MODE, NH>, dim3(p.HB, grid_cta), dim3(kThreads), smem, s, p);
  return launch_combine(c, p, s, e, ev);
}

cudaError_t launch_decode(mlaq_cache* c, const uint16_t* q_latent, const uint16_t* q_rope,
                          const int32_t* page_table, const int32_t* seq_lens, int B, int H, float scale,
                          uint16_t* out, float* lse, cudaStream_t s, int q_len) {
  char* ws = static_cast<char*>(c->workspace);
  const WsLayout lay = ws_layout(c->max_seqs, c->max_heads);
  // Kernel: the register-score kernel by default (measured faster on GB300
  // for every head count; the tcgen05-score kernel is variant 2), with 32
  // heads per CTA when H allows it (one unpack per page for both halves), 16
  // otherwise; the tcgen05-score kernel with 64, 32 or 16 heads per CTA.
  const bool tc = c->decode_variant == 2;
  const int NH = tc ? (H % 64 == 0 ? 64 : H % 32 == 0 ? 32 : 16) : (H % 32 == 0 ? 32 : 16);
  const int HB = H / NH;
  // item slots (CTAs per head block): by default one wave of the kernel's
  // resident CTAs (tcgen05 kernel: one per SM)
  const int ctas = c->decode_ctas_set ? c->decode_ctas
                   : tc              ? max(1, c->num_sms)
                                     : min(kMaxPlanCtas, (NH == 16 ? ctas_per_sm<16>() : ctas_per_sm<32>()) *
                                                              max(1, c->num_sms));
  const int G = plan_slots(ctas, HB, H);

  DecodeParams p;
  p.codes = static_cast<const uint8_t*>(c->codes);
  p.meta = static_cast<const uint8_t*>(c->meta);
  p.ring = static_cast<const uint16_t*>(c->ring);
  p.q_latent = q_latent;
  p.q_rope = q_rope;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.status = reinterpret_cast<int*>(ws + kWsStatus);
  p.items = reinterpret_cast<const Item*>(ws + lay.items);
  p.item_start = reinterpret_cast<const int*>(ws + lay.item_start);
  p.cta_item_start = reinterpret_cast<const int*>(ws + lay.cta_item_start);
  p.cta_first = reinterpret_cast<const Item*>(ws + lay.cta_first);
  p.o_part = reinterpret_cast<__half*>(ws + lay.o_part);
  p.lse_part = reinterpret_cast<float*>(ws + lay.lse_part);
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.HB = HB;
  p.q_len = q_len;
  p.h_per_q = H / q_len;
  p.max_pages = c->max_pages_per_seq;
  p.num_pages = c->num_pages;
  p.max_tokens = c->max_pages_per_seq * kPage;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.cost_step = c->cost_step;
  p.cost_ring = c->cost_ring;
  p.cost_item = c->cost_item;
  // Shares of the first, second and third resident CTA of an SM. Per-CTA
  // timing on GB300 (V2-Lite and serving C4R4 alike) gave 4.02, 4.24 and
  // 4.44 us per page for three 16-head CTAs per SM at equal shares, and the
  // later slots slow down further when they hold less: shares 1 : 0.925 :
  // 0.86 measured best (serving 194.4 us per call against 199.8 at equal
  // shares, V2-Lite 111.1 against 111.5). Two 32-head CTAs per SM differ by
  // 1%; one tcgen05 CTA per SM has one slot.
  p.sms = max(1, c->num_sms);
  const bool three = !tc && NH == 16;
  p.slot_w[0] = 1000;
  p.slot_w[1] = three ? 925 : 1000;
  p.slot_w[2] = three ? 860 : 1000;

  {
    const cudaError_t ea = decode_attrs_ready();
    if (ea != cudaSuccess) return ea;
  }
  // timed (mlaq_timing_enable): plan + decode + combine
  if (c->timing_events && c->timing_n < c->timing_max)
    cudaEventRecord(reinterpret_cast<cudaEvent_t*>(c->timing_events)[2 * c->timing_n], s);
  // one thread per sequence or CTA boundary (pass C scans G + 1 values in one
  // pass), in whole warps: small batches synchronise fewer warps
  const int plan_threads = min(1024, (max(B, G + 1) + 31) / 32 * 32);
  cudaError_t e = launch_pdl(plan_kernel, dim3(1), dim3(plan_threads), plan_smem_bytes(B, G), s, p, (int)c->mode, G,
                             reinterpret_cast<Item*>(ws + lay.items), reinterpret_cast<int*>(ws + lay.item_start),
                             reinterpret_cast<int*>(ws + lay.cta_item_start),
                             reinterpret_cast<Item*>(ws + lay.cta_first), reinterpret_cast<int*>(ws + kWsNumItems));
  if (e != cudaSuccess) return e;
  if (tc) {
    if (NH == 64) {
      if (c->mode == MLAQ_C4R4) return run_decode_tc<MLAQ_C4R4, 64>(c, p, G, s);
      if (c->mode == MLAQ_C2R4) return run_decode_tc<MLAQ_C2R4, 64>(c, p, G, s);
      return run_decode_tc<MLAQ_BF16, 64>(c, p, G, s);
    }
    if (NH == 32) {
      if (c->mode == MLAQ_C4R4) return run_decode_tc<MLAQ_C4R4, 32>(c, p, G, s);
      if (c->mode == MLAQ_C2R4) return run_decode_tc<MLAQ_C2R4, 32>(c, p, G, s);
      return run_decode_tc<MLAQ_BF16, 32>(c, p, G, s);
    }
    if (c->mode == MLAQ_C4R4) return run_decode_tc<MLAQ_C4R4, 16>(c, p, G, s);
    if (c->mode == MLAQ_C2R4) return run_decode_tc<MLAQ_C2R4, 16>(c, p, G, s);
    return run_decode_tc<MLAQ_BF16, 16>(c, p, G, s);
  }
  if (NH == 32) {
    if (c->mode == MLAQ_C4R4) return run_decode<MLAQ_C4R4, 32>(c, p, G, s);
    if (c->mode == MLAQ_C2R4) return run_decode<MLAQ_C2R4, 32>(c, p, G, s);
    return run_decode<MLAQ_BF16, 32>(c, p, G, s);
  }
  if (c->mode == MLAQ_C4R4) return run_decode<MLAQ_C4R4, 16>(c, p, G, s);
  if (c->mode == MLAQ_C2R4) return run_decode<MLAQ_C2R4, 16>(c, p, G, s);
  return run_decode<MLAQ_BF16, 16>(c, p, G, s);
}

size_t workspace_bytes_for(int max_seqs, int max_heads) { return ws_layout(max_seqs, max_heads).total; }

}  // namespace mlaq

// ---------------------------------------------------------------------------
// Allocation-free decode.
//
// For callers that cannot allocate device memory themselves: code running
// inside another runtime's allocator, a plugin that may not call cudaMalloc
// while a stream is being captured, or a host that pre-reserves all of HBM.
// The plan and the split partials normally live in the caller's workspace;
// here they live in a fixed array inside this library. The array is a
// file-scope __device__ variable, so every GPU that loads the library holds
// it until the process exits.
namespace mlaq {

constexpr size_t kStaticScratchBytes = (size_t)64 << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

static void* g_static_ptr[kMaxDevices];
static int g_static_sms[kMaxDevices];
static std::atomic<bool> g_static_ready[kMaxDevices];
static std::mutex g_static_mutex;

// Once per device, with that device current: the scratch array's device
// address (host code only sees a host-side stand-in for the symbol), the SM
// count the planner sizes the grid for, and every decode kernel variant's
// attributes (so that no later call on this device changes one, whatever its
// mode or head count). Serialised across host threads.
static cudaError_t static_scratch_setup(int dev) {
  if (g_static_ready[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (g_static_ready[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  cudaError_t e = decode_attrs_ready();
  if (e != cudaSuccess) return e;
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  g_static_sms[dev] = sms;
  g_static_ptr[dev] = p;
  g_static_ready[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

size_t static_scratch_bytes() { return kStaticScratchBytes; }

// Returns MLAQ_* status (argument errors) or MLAQ_ERR_CUDA.
int launch_decode_static(int mode, const void* codes, const void* meta, const void* ring, int num_pages,
                         int max_pages_per_seq, const uint16_t* q_latent, const uint16_t* q_rope,
                         const int32_t* page_table, const int32_t* seq_lens, int B, int H, float scale,
                         uint16_t* out, float* lse, int32_t* dev_status, cudaStream_t s) {
  if (workspace_bytes_for(B, H) > kStaticScratchBytes) return MLAQ_ERR_CAPACITY;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLAQ_ERR_CUDA;
  if (static_scratch_setup(dev) != cudaSuccess) return MLAQ_ERR_CUDA;
  mlaq_cache c = {};
  c.mode = mode;
  c.num_pages = num_pages;
  c.max_seqs = B;
  c.max_pages_per_seq = max_pages_per_seq;
  c.max_heads = H;
  c.codes = const_cast<void*>(codes);
  c.meta = const_cast<void*>(meta);
  c.ring = const_cast<void*>(ring);
  c.workspace = g_static_ptr[dev];
  c.workspace_bytes = kStaticScratchBytes;
  c.num_sms = g_static_sms[dev];
  c.cost_step = kDefCostStep;
  c.cost_ring = kDefCostRing;
  c.cost_item = kDefCostItem;
  char* ws = static_cast<char*>(c.workspace);
  // the status word is sticky: start each call from zero
  if (cudaMemsetAsync(ws + kWsStatus, 0, sizeof(int), s) != cudaSuccess) return MLAQ_ERR_CUDA;
  if (launch_decode(&c, q_latent, q_rope, page_table, seq_lens, B, H, scale, out, lse, s) != cudaSuccess)
    return MLAQ_ERR_CUDA;
  if (dev_status &&
      cudaMemcpyAsync(dev_status, ws + kWsStatus, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MLAQ_ERR_CUDA;
  return MLAQ_OK;
}

}  // namespace mlaq
