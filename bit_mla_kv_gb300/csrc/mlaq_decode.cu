// Split-KV MLA decode over the mixed-precision paged cache, its device-side
// planner and the log-sum-exp combine.
//
// QuantMLA (ai.info "Key Contributions" item 4; onedev.kr "어떻게 쓰나"):
// unpack + dequant fused into attention, packed pages and metadata staged
// apart from the reconstructed tiles, 4 sink + 128 recent tokens read from
// BF16, a single softmax over all valid tokens.
//
// Design (one CTA = one work item x 16 heads; 4 warps):
//  * Packed pages (codes + fp16 meta) are staged by bulk-copy (TMA) into a
//    4-deep shared-memory ring, one 64-token page per stage.
//  * Warp w owns content groups 2w, 2w+1 (channels 128w..128w+127) and RoPE
//    channels 16w..16w+15. Each step covers 16 tokens.
//  * Scores use exact integer codes as fp16 MMA operands: the tile computes
//    D_g[t,h] = sum_{c in g} q[t,c] * Q[h,c] per group g, then
//    S[t,h] = sum_g s[t,g] * D_g[t,h] + sum_g mn[t,g] * sum_{c in g} Q[h,c]
//    (the second sum is one more m16n8k16 MMA on hi/lo fp16 splits of the
//    per-group query sums). This keeps the score exact up to fp32 rounding.
//  * The four warps' partial scores are summed through shared memory; each
//    warp then runs the online softmax for 4 heads (exp2, lazily rescaled max)
//    and publishes P in fp16.
//  * Aggregation reuses the same registers: the codes are dequantized once to
//    fp16 (c = q*s + mn, one rounding), transposed in registers with
//    movmatrix, and fed to m16n8k16 MMAs against P: O[h, c] += P[h, t] c[t, c].
//    The dequantized tile never touches shared memory.
//  * BF16 tokens (ring and the all-BF16 cache) take the same path with
//    (s, mn) = (1, 0).
#include <math.h>

#include "mlaq_internal.cuh"

namespace mlaq {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 4;
constexpr int kT = 16;                             // tokens per step
constexpr int kBf16StageTok = 16;                  // tokens per BF16 stage
constexpr int kStageBytes = kPage * 288 + kMetaPage;  // 20736: max(C4R4 page + meta, 16 BF16 tokens)
constexpr int kSpStride = 20;                      // floats per row of partial scores [h][t]
constexpr int kPStride = 24;                       // halfs per row of P [h][t]
constexpr int kMinPagesPerSplit = 4;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kMaxDevices = 64;

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
  const int* num_items;
  float* o_part;
  float* lse_part;
  int B, H, max_pages, num_pages;
  float scale_log2;
};

struct __align__(16) DecodeSmem {
  uint8_t stage[kStages][kStageBytes];
  float sp[kWarps][16][kSpStride];   // partial scores, [warp][head][token]
  __half pr[16][kPStride];           // P, [head][token]
  float alpha[16];
  float fin_m[16];
  float fin_l[16];
  int stage_bad[kStages];
  uint64_t full[kStages];
};

// ---------------------------------------------------------------------------
// Planner: one CTA. Splits every sequence's packed range [4, L-128) (or the
// whole range in BF16 mode) into page-aligned chunks so that the decode grid
// has about `target_items` chunks in total, plus one ring item per sequence.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* seq_lens, int B, int mode, int target_items,
                                                    int max_tokens, Item* items, int* item_start,
                                                    int* num_items, int* status) {
  __shared__ int red[32];
  __shared__ int carry;
  const int tid = threadIdx.x;
  // pass 1: total pages
  int local = 0;
  for (int b = tid; b < B; b += blockDim.x) {
    int L = min(max(seq_lens[b], 0), max_tokens);
    local += (mode == MLAQ_BF16) ? (L + kPage - 1) / kPage : (L > kRing ? (L - kRecent + kPage - 1) / kPage : 0);
  }
  for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
  if ((tid & 31) == 0) red[tid >> 5] = local;
  if (tid == 0) carry = 0;
  __syncthreads();
  if (tid < 32) {
    int v = (tid < (int)(blockDim.x >> 5)) ? red[tid] : 0;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (tid == 0) red[0] = v;
  }
  __syncthreads();
  const int total_pages = red[0];
  const int target = max(kMinPagesPerSplit, (total_pages + target_items - 1) / max(target_items, 1));
  __syncthreads();
  // pass 2: item counts, block scan in chunks of blockDim, item emission
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + tid;
    int L = 0, n = 0, ring = 0, tlo = 0, thi = 0;
    if (b < B) {
      int Lraw = seq_lens[b];
      if (Lraw > max_tokens) atomicOr(status, MLAQ_DEV_SEQ_OVERFLOW);
      L = min(max(Lraw, 0), max_tokens);
      if (mode == MLAQ_BF16) {
        tlo = 0, thi = L;
        n = (L + kPage - 1) / kPage;
      } else {
        ring = L > 0;
        if (L > kRing) {
          tlo = kSink, thi = L - kRecent;
          n = (thi + kPage - 1) / kPage;
        }
      }
    }
    const int splits = n > 0 ? (n + target - 1) / target : 0;
    const int cnt = ring + splits;
    // inclusive warp scan then block scan
    int v = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, v, o);
      if ((tid & 31) >= o) v += u;
    }
    __syncthreads();
    if ((tid & 31) == 31) red[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
      int w = (tid < (int)(blockDim.x >> 5)) ? red[tid] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, w, o);
        if (tid >= o) w += u;
      }
      red[tid] = w;  // inclusive over warps
    }
    __syncthreads();
    const int warp_prefix = (tid >> 5) ? red[(tid >> 5) - 1] : 0;
    const int start = carry + warp_prefix + v - cnt;
    if (b < B) {
      item_start[b] = start;
      int k = start;
      if (ring) items[k++] = Item{b, 1, 0, L};
      for (int j = 0; j < splits; ++j) {
        int pa = (int)((long long)j * n / splits), pb = (int)((long long)(j + 1) * n / splits);
        items[k++] = Item{b, 0, max(tlo, pa * kPage), min(thi, pb * kPage)};
      }
    }
    __syncthreads();
    if (tid == 0) carry += red[(blockDim.x >> 5) - 1];
    __syncthreads();
  }
  if (tid == 0) {
    item_start[B] = carry;
    *num_items = carry;
  }
}

// ---------------------------------------------------------------------------
// Unpack helpers: fp16 pair (1024 + m*q) via LOP3, then exact q via HFMA2.
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, uint32_t mask, uint32_t inv_m, uint32_t neg_off) {
  uint32_t v = lop3_and_or(w, mask, 0x64006400u);
  return h2_as_u32(__hfma2(u32_as_h2(v), u32_as_h2(inv_m), u32_as_h2(neg_off)));
}
// fp16 constants as packed pairs
constexpr uint32_t kH1 = 0x3C003C00u;       // 1.0
constexpr uint32_t kHm1024 = 0xE400E400u;   // -1024
constexpr uint32_t kH1_4 = 0x34003400u;     // 0.25
constexpr uint32_t kHm256 = 0xDC00DC00u;    // -256
constexpr uint32_t kH1_16 = 0x2C002C00u;    // 0.0625
constexpr uint32_t kHm64 = 0xD400D400u;     // -64
constexpr uint32_t kH1_64 = 0x24002400u;    // 0.015625
constexpr uint32_t kHm16 = 0xCC00CC00u;     // -16

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

// Validity of token slot `pos` of a stage (absolute token index for paged
// items, ring slot index for ring items).
__device__ __forceinline__ bool token_valid(const Item& it, int pos) {
  if (it.kind == 0) return pos >= it.tlo && pos < it.thi;
  const int L = it.thi;
  if (pos >= kRing) return false;
  if (pos < kSink) return pos < L;
  const int r = pos - kSink;
  const int t = (L - 1) - (((L - 1 - r) % kRecent + kRecent) % kRecent);
  return L > 0 && t >= kSink;
}

template <int MODE>
struct StagePlan {
  // number of stages of an item and tokens per stage
  __device__ static int count(const Item& it) {
    if (it.kind == 1) return (kRing + kBf16StageTok - 1) / kBf16StageTok;
    if (MODE == MLAQ_BF16) return (it.thi + kBf16StageTok - 1) / kBf16StageTok - it.tlo / kBf16StageTok;
    return (it.thi + kPage - 1) / kPage - it.tlo / kPage;
  }
  __device__ static bool paged_packed(const Item& it) { return MODE != MLAQ_BF16 && it.kind == 0; }
  // first token position of stage k
  __device__ static int base(const Item& it, int k) {
    if (it.kind == 1) return k * kBf16StageTok;
    if (MODE == MLAQ_BF16) return (it.tlo / kBf16StageTok + k) * kBf16StageTok;
    return (it.tlo / kPage + k) * kPage;
  }
};

// Producer: issue the bulk copies of stage k into buffer `buf`.
template <int MODE>
__device__ void issue_stage(const DecodeParams& p, DecodeSmem& sm, const Item& it, int k, int buf) {
  uint64_t* bar = &sm.full[buf];
  const int base = StagePlan<MODE>::base(it, k);
  if (it.kind == 1) {
    const int n = min(kBf16StageTok, kRing - base);
    const uint32_t bytes = n * kD * 2;
    sm.stage_bad[buf] = 0;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(sm.stage[buf], p.ring + ((size_t)it.b * kRing + base) * kD, bytes, bar);
    return;
  }
  const int pidx = base / kPage;
  int page = -1;
  if (pidx < p.max_pages) page = p.page_table[(size_t)it.b * p.max_pages + pidx];
  if (page < 0 || page >= p.num_pages) {
    atomicOr(p.status, MLAQ_DEV_PAGE_OOB);
    sm.stage_bad[buf] = 1;
    mbar_arrive_expect_tx(bar, 0);
    return;
  }
  sm.stage_bad[buf] = 0;
  if constexpr (MODE == MLAQ_BF16) {
    const uint32_t bytes = kBf16StageTok * kD * 2;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(sm.stage[buf], p.codes + (size_t)page * page_code_bytes(MODE) + (size_t)(base % kPage) * kD * 2,
             bytes, bar);
  } else {
    const uint32_t cb = page_code_bytes(MODE);
    mbar_arrive_expect_tx(bar, cb + kMetaPage);
    bulk_g2s(sm.stage[buf], p.codes + (size_t)page * cb, cb, bar);
    bulk_g2s(sm.stage[buf] + cb, p.meta + (size_t)page * kMetaPage, kMetaPage, bar);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
  // head blocks of one item are adjacent in launch order so they share L2
  const int item_idx = blockIdx.y;
  if (item_idx >= *p.num_items) return;
  const Item it = p.items[item_idx];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, i = lane & 3;
  const int h0 = blockIdx.x * 16;
  const int nst = StagePlan<MODE>::count(it);
  constexpr int CB = token_bytes(MODE);
  constexpr int CBITS = content_bits(MODE);
  constexpr int GBYTES = group_code_bytes(CBITS);
  constexpr int ROPE_OFF = 8 * GBYTES;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], 1);
    fence_mbar_init();
    fence_proxy_async();
  }
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < min(kStages, nst); ++k) issue_stage<MODE>(p, sm, it, k, k);

  // ---- query fragments (B operand of the score MMA: k = channel, n = head)
  // qf[j][kk][hb][0..1], j: content group 2w+j; rope: qr[hb][0..1]
  uint32_t qf[2][4][2][2], qr[2][2];
  float k2[3][2];  // per-group query sums for heads r (hb=0) and r+8 (hb=1)
  {
    const uint16_t* ql = p.q_latent + ((size_t)it.b * p.H + h0) * kDL;
    const uint16_t* qp = p.q_rope + ((size_t)it.b * p.H + h0) * kDR;
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int h = 8 * hb + r;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float acc = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int c = 64 * (2 * w + j) + 16 * kk + 2 * i;
          uint32_t u0 = *reinterpret_cast<const uint32_t*>(ql + (size_t)h * kDL + c);
          uint32_t u1 = *reinterpret_cast<const uint32_t*>(ql + (size_t)h * kDL + c + 8);
          qf[j][kk][hb][0] = bf2_to_h2(u0);
          qf[j][kk][hb][1] = bf2_to_h2(u1);
          float2 a = __half22float2(u32_as_h2(qf[j][kk][hb][0]));
          float2 bq = __half22float2(u32_as_h2(qf[j][kk][hb][1]));
          acc += (a.x + a.y) + (bq.x + bq.y);
        }
        k2[j][hb] = acc;
      }
      {
        const int c = 16 * w + 2 * i;
        uint32_t u0 = *reinterpret_cast<const uint32_t*>(qp + (size_t)h * kDR + c);
        uint32_t u1 = *reinterpret_cast<const uint32_t*>(qp + (size_t)h * kDR + c + 8);
        qr[hb][0] = bf2_to_h2(u0);
        qr[hb][1] = bf2_to_h2(u1);
        float2 a = __half22float2(u32_as_h2(qr[hb][0]));
        float2 bq = __half22float2(u32_as_h2(qr[hb][1]));
        k2[2][hb] = (a.x + a.y) + (bq.x + bq.y);
      }
    }
  }
  // quad reduction of the query sums (the 4 lanes i share head r)
#pragma unroll
  for (int j = 0; j < 3; ++j)
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      float v = k2[j][hb];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      k2[j][hb] = v;
    }
  // B fragment of the min-term MMA: rows k = 2j, 2j+1 hold hi/lo of K2_j.
  uint32_t kmn[2];
#pragma unroll
  for (int hb = 0; hb < 2; ++hb) {
    float v = (i == 0) ? k2[0][hb] : (i == 1) ? k2[1][hb] : k2[2][hb];
    __half hi = __float2half_rn(v);
    __half lo = __float2half_rn(v - __half2float(hi));
    kmn[hb] = (i < 3) ? h2_as_u32(__halves2half2(hi, lo)) : 0u;
  }

  float o[2][4][2][4];  // [j][kk][cb][4]: O[h = r / r+8][c = 64(2w+j) + 16kk + 8cb + 2i..]
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int cb = 0; cb < 2; ++cb)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[j][kk][cb][e] = 0.f;

  // softmax state of the reducer lanes: head hh = 4w + lane/8, tokens 2*(lane%8)..+1
  const int hh = 4 * w + (lane >> 3);
  const int tp = 2 * (lane & 7);
  float m_run = -INFINITY, l_run = 0.f;
  bool failed = false;
  int k_fail = 0;

  for (int k = 0; k < nst && !failed; ++k) {
    const int buf = k % kStages;
    const bool ok = mbar_wait_bounded(&sm.full[buf], (k / kStages) & 1, kWaitLimit);
    const uint8_t* st = sm.stage[buf];
    const bool bad = sm.stage_bad[buf] != 0;
    const int base = StagePlan<MODE>::base(it, k);
    const bool packed = StagePlan<MODE>::paged_packed(it);
    const int nsteps = packed ? kPage / kT : 1;
    for (int s = 0; s < nsteps; ++s) {
      const int tb = base + s * kT;
      const int lr = s * kT + r;  // local row of token r in the stage
      // every token of the step valid (the common case inside a packed range)
      const bool all_in = it.kind == 0 && tb >= it.tlo && tb + kT <= it.thi;
      const bool v0 = ok && !bad && (all_in || token_valid(it, tb + r));
      const bool v1 = ok && !bad && (all_in || token_valid(it, tb + 8 + r));
      // ---------------- dequant + scores
      // meta for tokens r (x) and r+8 (y), groups j = 0, 1 (content), 2 (rope)
      uint32_t mx[3], my[3];
      uint32_t ch[2][4][4];  // fp16 A fragments of the content tile (exact codes, later dequantized)
      float sacc[2][4];      // S[t][h] for head blocks 0/1
#pragma unroll
      for (int hb = 0; hb < 2; ++hb)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[hb][e] = 0.f;
      uint32_t rf[4];
      if (packed) {
        const uint8_t* mtab = st + page_code_bytes(MODE);
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int g = j < 2 ? 2 * w + j : 8;
          mx[j] = v0 ? *reinterpret_cast<const uint32_t*>(mtab + lr * kMetaTok + 4 * g) : 0u;
          my[j] = v1 ? *reinterpret_cast<const uint32_t*>(mtab + (lr + 8) * kMetaTok + 4 * g) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int g = 2 * w + j;
          if (CBITS == 4) {
            uint2 wx = *reinterpret_cast<const uint2*>(st + lr * CB + g * GBYTES + 8 * i);
            uint2 wy = *reinterpret_cast<const uint2*>(st + (lr + 8) * CB + g * GBYTES + 8 * i);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              uint32_t ax = (kk >> 1) ? wx.y : wx.x, ay = (kk >> 1) ? wy.y : wy.x;
              uint32_t ax8 = ax >> 8, ay8 = ay >> 8;
              const int p0 = 2 * (kk & 1);
              ch[j][kk][0] = int4_pos(ax, ax8, p0);
              ch[j][kk][1] = int4_pos(ay, ay8, p0);
              ch[j][kk][2] = int4_pos(ax, ax8, p0 + 1);
              ch[j][kk][3] = int4_pos(ay, ay8, p0 + 1);
            }
          } else {
            uint32_t ax = *reinterpret_cast<const uint32_t*>(st + lr * CB + g * GBYTES + 4 * i);
            uint32_t ay = *reinterpret_cast<const uint32_t*>(st + (lr + 8) * CB + g * GBYTES + 4 * i);
            uint32_t ax8 = ax >> 8, ay8 = ay >> 8;
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
          if (i & 1) { ax >>= 8; ay >>= 8; }
          rf[0] = int4_pos(ax, 0u, 0);
          rf[1] = int4_pos(ay, 0u, 0);
          rf[2] = int4_pos(ax, 0u, 1);
          rf[3] = int4_pos(ay, 0u, 1);
        }
      } else {
        // BF16 tokens (ring or all-BF16 pages): q = x, (s, mn) = (1, 0)
        const uint32_t one = 0x00003C00u;  // (s = 1, mn = 0)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          mx[j] = v0 ? one : 0u;
          my[j] = v1 ? one : 0u;
        }
        const uint8_t* rx = st + lr * (kD * 2);
        const uint8_t* ry = st + (lr + 8) * (kD * 2);
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int c = 64 * (2 * w + j) + 16 * kk + 2 * i;
            ch[j][kk][0] = v0 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(rx + 2 * c)) : 0u;
            ch[j][kk][1] = v1 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(ry + 2 * c)) : 0u;
            ch[j][kk][2] = v0 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(rx + 2 * c + 16)) : 0u;
            ch[j][kk][3] = v1 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(ry + 2 * c + 16)) : 0u;
          }
        const int c = kDL + 16 * w + 2 * i;
        rf[0] = v0 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(rx + 2 * c)) : 0u;
        rf[1] = v1 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(ry + 2 * c)) : 0u;
        rf[2] = v0 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(rx + 2 * c + 16)) : 0u;
        rf[3] = v1 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(ry + 2 * c + 16)) : 0u;
      }
      // min term: S += [mn_j hi-lo rows] . [K2_j hi, lo]
      {
        uint32_t a[4];
        uint32_t mnx = (i == 0) ? mx[0] : (i == 1) ? mx[1] : mx[2];
        uint32_t mny = (i == 0) ? my[0] : (i == 1) ? my[1] : my[2];
        // (mn, mn) pairs: high halves of the meta words
        a[0] = (i < 3) ? __byte_perm(mnx, 0, 0x3232) : 0u;
        a[1] = (i < 3) ? __byte_perm(mny, 0, 0x3232) : 0u;
        a[2] = 0u;
        a[3] = 0u;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) mma16816(sacc[hb], a, kmn[hb], 0u);
      }
      // scale terms per group
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        float d[2][4];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb)
#pragma unroll
          for (int e = 0; e < 4; ++e) d[hb][e] = 0.f;
        if (j < 2) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              uint32_t bq0 = qf[j][kk][hb][0], bq1 = qf[j][kk][hb][1];
              mma16816(d[hb], ch[j][kk], bq0, bq1);
            }
        } else {
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) mma16816(d[hb], rf, qr[hb][0], qr[hb][1]);
        }
        const float sx = __half2float(__ushort_as_half((unsigned short)(mx[j] & 0xffffu)));
        const float sy = __half2float(__ushort_as_half((unsigned short)(my[j] & 0xffffu)));
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          sacc[hb][0] = fmaf(sx, d[hb][0], sacc[hb][0]);
          sacc[hb][1] = fmaf(sx, d[hb][1], sacc[hb][1]);
          sacc[hb][2] = fmaf(sy, d[hb][2], sacc[hb][2]);
          sacc[hb][3] = fmaf(sy, d[hb][3], sacc[hb][3]);
        }
      }
      // publish partial scores: sacc[hb] = S[t = r (e 0,1) / r+8 (e 2,3)][h = 8hb + 2i (+1)]
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int h = 8 * hb + 2 * i;
        sm.sp[w][h][r] = sacc[hb][0];
        sm.sp[w][h + 1][r] = sacc[hb][1];
        sm.sp[w][h][r + 8] = sacc[hb][2];
        sm.sp[w][h + 1][r + 8] = sacc[hb][3];
      }
      // dequantize the content tile in place (fp16, one rounding) and
      // transpose each 8x8 block for the aggregation B operand.
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const __half2 s2x = __low2half2(u32_as_h2(mx[j])), m2x = __high2half2(u32_as_h2(mx[j]));
        const __half2 s2y = __low2half2(u32_as_h2(my[j])), m2y = __high2half2(u32_as_h2(my[j]));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          ch[j][kk][0] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][0]), s2x, m2x)));
          ch[j][kk][1] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][1]), s2y, m2y)));
          ch[j][kk][2] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][2]), s2x, m2x)));
          ch[j][kk][3] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][3]), s2y, m2y)));
        }
      }
      // barrier 1: partial scores complete; also agrees on a timed-out wait
      const bool any_fail = named_bar_or(1, kThreads, !ok);
      if (any_fail) {
        failed = true;
        k_fail = k;
        break;
      }
      // the stage's shared memory is no longer read: refill it
      if (tid == 0 && s == nsteps - 1 && k + kStages < nst) issue_stage<MODE>(p, sm, it, k + kStages, buf);
      // ---------------- online softmax for head hh, tokens tp, tp+1
      {
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) {
          float2 v = *reinterpret_cast<const float2*>(&sm.sp[ww][hh][tp]);
          x0 += v.x;
          x1 += v.y;
        }
        const bool ok0 = !bad && (all_in || token_valid(it, tb + tp));
        const bool ok1 = !bad && (all_in || token_valid(it, tb + tp + 1));
        x0 = ok0 ? x0 * p.scale_log2 : -INFINITY;
        x1 = ok1 ? x1 * p.scale_log2 : -INFINITY;
        float tmax = fmaxf(x0, x1);
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
        float alpha = 1.f;
        if (tmax > m_run + 8.f) {  // lazy rescale: keep a stale max while P <= 2^8
          alpha = ex2(m_run - tmax);  // m_run = -inf gives 0
          m_run = tmax;
        }
        const float mref = (m_run == -INFINITY) ? 0.f : m_run;  // all-masked so far: x = -inf -> p = 0
        const float p0 = ex2(x0 - mref), p1 = ex2(x1 - mref);
        l_run = l_run * alpha + (p0 + p1);
        *reinterpret_cast<__half2*>(&sm.pr[hh][tp]) = __floats2half2_rn(p0, p1);
        if ((lane & 7) == 0) sm.alpha[hh] = alpha;
      }
      named_bar_sync(2, kThreads);
      // ---------------- aggregation
      {
        const float ar = sm.alpha[r], ar8 = sm.alpha[r + 8];
        if (__any_sync(0xffffffffu, ar != 1.f || ar8 != 1.f)) {
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
              for (int cb = 0; cb < 2; ++cb) {
                o[j][kk][cb][0] *= ar;
                o[j][kk][cb][1] *= ar;
                o[j][kk][cb][2] *= ar8;
                o[j][kk][cb][3] *= ar8;
              }
        }
        uint32_t pa[4];
        {
          const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
          const int col = 8 * (lane >> 4);
          ldmatrix_x4(pa, &sm.pr[row][col]);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // channel block cb = 0: B = (movmatrix of a0, a1); cb = 1: (a2, a3)
            mma16816(o[j][kk][0], pa, ch[j][kk][0], ch[j][kk][1]);
            mma16816(o[j][kk][1], pa, ch[j][kk][2], ch[j][kk][3]);
          }
      }
      // no barrier needed before the next step's writes to sp: every thread
      // passed barrier 2 after all reads of sp; pr/alpha are rewritten only
      // after the next barrier 1, which all threads reach after their reads.
    }
  }

  if (failed) {
    if (tid == 0) {
      atomicOr(p.status, MLAQ_DEV_TIMEOUT);
      // wait (bounded) for copies still in flight before the CTA exits
      for (int kk = k_fail; kk < min(nst, k_fail + kStages); ++kk)
        mbar_wait_bounded(&sm.full[kk % kStages], (kk / kStages) & 1, kWaitLimit);
    }
  }
  // ---- finalize: reduce l over the 8 lanes of each head
  float l_tot = l_run;
  l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
  l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
  l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 4);
  if ((lane & 7) == 0) {
    sm.fin_m[hh] = m_run;
    sm.fin_l[hh] = failed ? 0.f : l_tot;
  }
  __syncthreads();
  const int H = p.H;
  float* op = p.o_part + ((size_t)item_idx * H + h0) * kDL;
  {
    const float lr0 = sm.fin_l[r], lr8 = sm.fin_l[r + 8];
    const float inv0 = lr0 > 0.f ? 1.f / lr0 : 0.f, inv8 = lr8 > 0.f ? 1.f / lr8 : 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          const int c = 64 * (2 * w + j) + 16 * kk + 8 * cb + 2 * i;
          *reinterpret_cast<float2*>(op + (size_t)r * kDL + c) =
              make_float2(o[j][kk][cb][0] * inv0, o[j][kk][cb][1] * inv0);
          *reinterpret_cast<float2*>(op + (size_t)(r + 8) * kDL + c) =
              make_float2(o[j][kk][cb][2] * inv8, o[j][kk][cb][3] * inv8);
        }
  }
  if (tid < 16) {
    const float l = sm.fin_l[tid];
    p.lse_part[(size_t)item_idx * H + h0 + tid] =
        l > 0.f ? (sm.fin_m[tid] + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// Combine: one warp per (b, h); log-sum-exp merge of the item partials.
__global__ void combine_kernel(const float* o_part, const float* lse_part, const int* item_start, int B, int H,
                               uint16_t* out, float* lse) {
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= B * H) return;
  const int b = gw / H, h = gw % H;
  const int s0 = item_start[b], s1 = item_start[b + 1];
  float m = -INFINITY;
  for (int s = s0; s < s1; ++s) m = fmaxf(m, lse_part[(size_t)s * H + h]);
  float4 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  float tot = 0.f;
  if (m != -INFINITY) {
    for (int s = s0; s < s1; ++s) {
      const float ls = lse_part[(size_t)s * H + h];
      const float wgt = expf(ls - m);
      tot += wgt;
      if (wgt == 0.f) continue;
      const float4* src = reinterpret_cast<const float4*>(o_part + ((size_t)s * H + h) * kDL);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float4 v = src[lane + 32 * q];
        acc[q].x += wgt * v.x;
        acc[q].y += wgt * v.y;
        acc[q].z += wgt * v.z;
        acc[q].w += wgt * v.w;
      }
    }
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  uint16_t* dst = out + ((size_t)b * H + h) * kDL;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = 4 * (lane + 32 * q);
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[q].x * inv, acc[q].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[q].z * inv, acc[q].w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst + c) = pk;
  }
  if (lane == 0) lse[(size_t)b * H + h] = tot > 0.f ? m + logf(tot) : -INFINITY;
}

// ---------------------------------------------------------------------------
template <int MODE>
static cudaError_t run_decode(mlaq_cache* c, const DecodeParams& p, int grid_x, int grid_y, cudaStream_t s) {
  const int smem = (int)sizeof(DecodeSmem);
  // Opt in to >48 KB of dynamic shared memory once per device (the first call
  // on a device must not be inside a stream capture).
  static bool attr_done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t ea = cudaGetDevice(&dev);
  if (ea != cudaSuccess) return ea;
  if (dev < 0 || dev >= kMaxDevices || !attr_done[dev]) {
    ea = cudaFuncSetAttribute(decode_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (ea != cudaSuccess) return ea;
    if (dev >= 0 && dev < kMaxDevices) attr_done[dev] = true;
  }
  cudaEvent_t* ev = nullptr;
  if (c->timing_events && c->timing_n < c->timing_max) {
    ev = reinterpret_cast<cudaEvent_t*>(c->timing_events) + 2 * c->timing_n;
    cudaEventRecord(ev[0], s);
  }
  decode_kernel<MODE><<<dim3(grid_y, grid_x), kThreads, smem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (ev) {
    cudaEventRecord(ev[1], s);
    c->timing_n++;
  }
  return e;
}

cudaError_t launch_decode(mlaq_cache* c, const uint16_t* q_latent, const uint16_t* q_rope,
                          const int32_t* page_table, const int32_t* seq_lens, int B, int H, float scale,
                          uint16_t* out, float* lse, cudaStream_t s) {
  char* ws = static_cast<char*>(c->workspace);
  const size_t max_items = max_items_for(c->max_seqs);
  Item* items = reinterpret_cast<Item*>(ws + kWsItems);
  int* item_start = reinterpret_cast<int*>(ws + kWsItems + max_items * sizeof(Item));
  size_t off = kWsItems + max_items * sizeof(Item) + ((size_t)(c->max_seqs + 1) * 4 + 255) / 256 * 256;
  float* lse_part = reinterpret_cast<float*>(ws + off);
  off += (max_partial_rows(c->max_seqs, c->max_heads) * 4 + 255) / 256 * 256;
  float* o_part = reinterpret_cast<float*>(ws + off);
  int* status = reinterpret_cast<int*>(ws + kWsStatus);
  int* num_items = reinterpret_cast<int*>(ws + kWsNumItems);

  const int head_blocks = H / 16;
  const int target_items = max(1, min(kMaxPlanCtas, c->decode_ctas / head_blocks));
  const int max_tokens = c->max_pages_per_seq * kPage;
  plan_kernel<<<1, 1024, 0, s>>>(seq_lens, B, c->mode, target_items, max_tokens, items, item_start, num_items,
                                 status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  DecodeParams p;
  p.codes = static_cast<const uint8_t*>(c->codes);
  p.meta = static_cast<const uint8_t*>(c->meta);
  p.ring = static_cast<const uint16_t*>(c->ring);
  p.q_latent = q_latent;
  p.q_rope = q_rope;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.status = status;
  p.items = items;
  p.num_items = num_items;
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.B = B;
  p.H = H;
  p.max_pages = c->max_pages_per_seq;
  p.num_pages = c->num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int grid_x = (int)min((size_t)(2 * B + target_items), max_items);
  if (c->mode == MLAQ_C4R4) e = run_decode<MLAQ_C4R4>(c, p, grid_x, head_blocks, s);
  else if (c->mode == MLAQ_C2R4) e = run_decode<MLAQ_C2R4>(c, p, grid_x, head_blocks, s);
  else e = run_decode<MLAQ_BF16>(c, p, grid_x, head_blocks, s);
  if (e != cudaSuccess) return e;
  const int warps = B * H;
  combine_kernel<<<(warps + 7) / 8, 256, 0, s>>>(o_part, lse_part, item_start, B, H, out, lse);
  return cudaGetLastError();
}

size_t workspace_bytes_for(int max_seqs, int max_heads) {
  const size_t max_items = max_items_for(max_seqs);
  size_t off = kWsItems + max_items * sizeof(Item) + ((size_t)(max_seqs + 1) * 4 + 255) / 256 * 256;
  off += (max_partial_rows(max_seqs, max_heads) * 4 + 255) / 256 * 256;
  off += max_partial_rows(max_seqs, max_heads) * kDL * 4;
  return off;
}

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

// Once per device, with that device current: the scratch array's device
// address (host code only sees a host-side stand-in for the symbol) and the
// SM count the planner sizes the grid for.
static cudaError_t static_scratch_setup(int dev) {
  if (g_static_ptr[dev]) return cudaSuccess;
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  g_static_sms[dev] = sms;
  g_static_ptr[dev] = p;
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
  c.decode_ctas = 2 * c.num_sms < kMaxPlanCtas ? 2 * c.num_sms : kMaxPlanCtas;
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
