// Split-KV MLA decode with both contractions on tcgen05 (included by
// mlaq_decode.cu: it shares the planner, the work items, the stage helpers
// and the combine kernel with the register-score kernel there).
//
// QuantMLA (ai.info "Key Contributions" item 4; onedev.kr "어떻게 쓰나"):
// unpack + dequant fused into attention, BF16 sink/recent tokens and packed
// tokens under one softmax, packed data and metadata staged apart from the
// reconstructed tiles so that prefetch overlaps the math.
//
// One CTA serves NH heads (16, 32 or 64) of one item at a time and walks its
// items' stages (packed pages, ring chunks, BF16 page quarters) in tiles of
// up to 128 rows (tokens).
//
// Scores on tcgen05, exact. With tokens on M (the 128 TMEM lanes) and heads
// on N, S[t, h] = sum_c Q[h, c] * c_hat[t, c] with c_hat = q * s + mn per
// 64-channel group. Each fp16 scale is split as s = s_hi + s_lo, s_hi being
// s with its four lowest mantissa bits cleared: with centered codes
// u = q - C (C = 8 for 4-bit, 2 for 2-bit codes), u * s_hi (4 x 7
// significant bits) and u * s_lo (4 x 4 bits) are exact fp16 values for
// every code and every fp16 scale, so with the group midpoint d = mn + C s
//   S = Q . [u s_hi] + Q . [u s_lo] + sum_g d_g * sum_{c in g} Q[h, c]
// is the exact score up to fp32 accumulation (and the centering keeps the
// accumulator near the size of S), computed by MMAs into one TMEM
// accumulator: A = the [u s_hi | u s_lo] tile of a group in TMEM (one
// thread per token writes its row), B = the query in shared memory; the
// midpoint term is one more K = 32 MMA on fp16 hi/lo splits of d and of the
// group sums of the query.
// (Rounding c_hat to fp16 instead gives lse errors up to 2e-3 on the
// outlier channels of the synthetic caches, over the 1e-3 bar.) BF16 rows
// (ring, all-BF16 cache) use their values as the hi part (lo = mn = 0).
//
// Aggregation on tcgen05 as in the register-score kernel: value warps unpack
// the content codes in MMA-fragment order, dequantize (fp16), transpose the
// 8x8 blocks with movmatrix and store V^T to TMEM (lanes = channels); one
// MMA per 16-token row group and 128-channel block accumulates O^T += V^T
// P^T in TMEM, B = P^T in shared memory.
//
// Roles (warp-specialized, mbarrier hand-offs, every wait bounded):
//   score warps (4 or 8)   score operands, softmax (one thread per token row;
//                          with 64 heads two warps per TMEM quadrant split
//                          each group's columns and the heads), P^T, lse
//   value warps (4)        V^T, lazy O^T rescale, epilogue
//   producer (1 lane)      bulk copies of stages into the shared-memory ring
//   score issuer (1 lane)  score MMAs
//   aggregation issuer     aggregation MMAs
namespace mlaq {

template <int NH>
struct TcCfg {
  static constexpr int SWQ = NH == 64 ? 2 : 1;  // score warps per TMEM lane quadrant
  static constexpr int HPW = NH / SWQ;          // heads per score warp
  static constexpr int kSW = 4 * SWQ;           // score warps
  static constexpr int kWarps = kSW + 4 + 3;    // + value warps, producer, two MMA issuers
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int wProd = kSW + 4, wSIss = kSW + 5, wAIss = kSW + 6;
  static constexpr int NA = NH == 64 ? 2 : 3;   // score operand columns: NA x 64
  // Score operand slots of the hand-off: a whole group (64 columns: hi 32 |
  // lo 32), written by every score warp (column half s of it when two warps
  // share a quadrant). (Half-group slots, one set per warp half, measured
  // slower: twice the hand-offs for no gain in overlap.)
  static constexpr int NAS = NA;
  static constexpr int kSlotCols = 64;
  static constexpr int NV = NH == 64 ? 2 : 4;   // V^T slots (32 columns: 4 blocks x 16 tokens)
  static constexpr int NS = NH == 64 ? 1 : 2;   // score accumulators
  static constexpr int NP = 2;                  // P^T buffers
  static constexpr int NSTG = NH == 64 ? 5 : 7; // stage buffers
  static constexpr uint32_t colO = 0, colS = 4 * NH, colA = colS + NS * NH, colV = colA + 64 * NA;
  static constexpr uint32_t kCols = 512;
  static_assert(colV + 32 * NV <= kCols, "TMEM columns");
  // Query blocks (B of the score MMAs): per (group, 16-channel step) NH heads
  // x 16 channels, K-major 8x16 B core matrices, k-core stride 128 B, n-core
  // stride 256 B.
  static constexpr int kQBlk = 32 * NH;
  // P^T (B of the aggregation MMAs), per 16-token row group: k-core stride
  // 144 B, n-core stride 288 B, row groups 32 B apart beyond that: the padding
  // spreads the 2-byte stores of a warp (one token row per lane, one head at
  // a time) over distinct banks.
  static constexpr int kPtLbo = 144, kPtSbo = 288;
  static constexpr int kPtRg = (NH / 8) * kPtSbo + 32;
  static constexpr int kMaxTileStages = 4;  // stages one tile may hold (ring chunks: 4 x 16 rows)
};

template <int NH>
struct __align__(128) TcSmem {
  using C = TcCfg<NH>;
  static constexpr int kNumStages = C::NSTG;
  uint8_t stage[C::NSTG][kStageBytes];
  __align__(128) uint8_t q[36 * C::kQBlk];       // query, [group][16-channel step] blocks
  __align__(128) uint8_t qm[2 * C::kQBlk];       // min term: K = 32 (hi, lo of 9 group sums, zero pad)
  __align__(128) uint8_t pt[C::NP][8 * C::kPtRg];
  uint64_t full[C::NSTG], empty[C::NSTG];
  uint64_t a_full[C::NAS], a_empty[C::NAS], s_full[C::NS], s_empty[C::NS];
  uint64_t v_full[C::NV], v_empty[C::NV], p_full[C::NP], p_empty[C::NP], o_free;
  int stage_bad[C::NSTG];
  uint32_t tmem_base;
  int abort;
  int vote[2][C::kSW];
  int rs_flag[C::NP][2];
  float m_run[NH];
  float alpha[C::NP][NH];
  float red[2][4][NH];
  float fin_m[2][NH], fin_l[2][NH];
};
static_assert(sizeof(TcSmem<64>) <= 227 * 1024 && sizeof(TcSmem<32>) <= 227 * 1024 &&
                  sizeof(TcSmem<16>) <= 227 * 1024,
              "tcgen05 decode shared memory");

// A bounded wait that gives up at once after any role of the CTA timed out
// (the CTA then runs to its end on whatever the buffers hold, so that every
// named barrier is still reached, and reports MLAQ_DEV_TIMEOUT).
template <class SM>
__device__ __forceinline__ void tc_wait(SM& sm, uint64_t* bar, uint32_t parity, int* status) {
  if (*reinterpret_cast<volatile int*>(&sm.abort)) return;
  if (!mbar_wait_bounded_sleep(bar, parity, kWaitLimit)) {
    *reinterpret_cast<volatile int*>(&sm.abort) = 1;
    atomicOr(status, MLAQ_DEV_TIMEOUT);
  }
}

// Uses of slot `slot` so far (a register array indexed by a runtime value
// through an unrolled select, so that it stays in registers).
template <int N>
__device__ __forceinline__ int tc_get(const int (&a)[N], int slot) {
  int v = 0;
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (k == slot) v = a[k];
  return v;
}
template <int N>
__device__ __forceinline__ void tc_bump(int (&a)[N], int slot) {
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (k == slot) a[k]++;
}

// Tiles of an item: runs of consecutive stages of at most 128 rows and
// kMaxTileStages stages (a packed page is 64 rows, a ring chunk or BF16 page
// quarter 16).
template <int MODE>
__device__ __forceinline__ int tc_tile_end(const Item& it, int L, int k0, int nst) {
  int rows = 0, k = k0;
  while (k < nst && k - k0 < TcCfg<16>::kMaxTileStages) {
    const int r = item_stage<MODE>(it, L, k).kind == 1 ? kPage : kT;
    if (rows + r > 128) break;
    rows += r;
    ++k;
  }
  return k;
}
template <int MODE>
__device__ __forceinline__ bool tc_tile_bf16(const Item& it, int L, int k0, int k1) {
  for (int k = k0; k < k1; ++k)
    if (item_stage<MODE>(it, L, k).kind == 1) return false;
  return true;
}

// Column pair k (channels 2k, 2k+1 of a group) of the code word wi, nibble
// position pp, in the physical layout (content_code_bit / rope_code_bit).
__host__ __device__ constexpr int tc_col_int4(int wi, int pp) {
  return 8 * (2 * (wi & 1) + (pp >> 1)) + 4 * (pp & 1) + (wi >> 1);
}
__host__ __device__ constexpr int tc_col_rope(int wi, int pp) {
  return 8 * (wi >> 1) + 4 * (pp & 1) + 2 * (wi & 1) + (pp >> 1);
}
__host__ __device__ constexpr int tc_col_int2(int wi, int pp) { return 8 * (pp >> 1) + 4 * (pp & 1) + wi; }
__host__ __device__ constexpr bool tc_cols_match_layout() {
  for (int wi = 0; wi < 8; ++wi)
    for (int pp = 0; pp < 4; ++pp)
      for (int ln = 0; ln < 2; ++ln) {
        if (content_code_bit(2 * tc_col_int4(wi, pp) + ln, 4) != wi * 32 + 16 * ln + 4 * pp) return false;
        if (rope_code_bit(2 * tc_col_rope(wi, pp) + ln) != wi * 32 + 16 * ln + 4 * pp) return false;
      }
  for (int wi = 0; wi < 4; ++wi)
    for (int pp = 0; pp < 8; ++pp)
      for (int ln = 0; ln < 2; ++ln)
        if (content_code_bit(2 * tc_col_int2(wi, pp) + ln, 2) != wi * 32 + 16 * ln + 2 * (pp & 3) + 8 * (pp >> 2))
          return false;
  return true;
}
static_assert(tc_cols_match_layout(), "score unpack columns must follow the physical code layout");

// K position of token t (0..15) of a row group in the V^T columns (the token
// order movmatrix leaves in the aggregation operand).
__device__ __forceinline__ int tc_kpos(int t) { return 4 * ((t & 7) >> 1) + 2 * (t >> 3) + (t & 1); }

// ---------------------------------------------------------------------------
// Producer: the CTA's stages in order, each into the next ring buffer once
// both consumer roles released it.
template <int MODE, int NH>
__device__ void tc_producer(const DecodeParams& p, TcSmem<NH>& sm, int cta, int i0, int i1) {
  using C = TcCfg<NH>;
  ProdCursor pc;
  producer_init<MODE>(p, pc, p.cta_first[cta], i0, i1);
  int n = 0;
  while (pc.item < i1) {
    if (n >= C::NSTG) {
      tc_wait(sm, &sm.empty[n % C::NSTG], ((n / C::NSTG) - 1) & 1, p.status);
      if (*reinterpret_cast<volatile int*>(&sm.abort)) break;
    }
    producer_advance<MODE>(p, sm, pc, i1);
    ++n;
  }
  // copies still in flight land before the CTA exits
  for (int k = max(0, n - C::NSTG); k < n; ++k) mbar_wait_bounded(&sm.full[k % C::NSTG], (k / C::NSTG) & 1, kWaitLimit);
}

// Score issuer: per tile, 4 MMAs (K = 16) per group on the hi operand, 4 on
// the lo operand, 2 for the min term, into the tile's score accumulator.
template <int MODE, int NH>
__device__ void tc_score_issuer(const DecodeParams& p, TcSmem<NH>& sm, uint32_t tmem, int i0, int i1) {
  using C = TcCfg<NH>;
  constexpr uint32_t idesc = umma_idesc_f16(128, NH);
  int a_use[C::NAS];
#pragma unroll
  for (int k = 0; k < C::NAS; ++k) a_use[k] = 0;
  int tile = 0;
  // descriptors of the first query block and of the min-term block; one
  // block further is kQBlk bytes, i.e. kQBlk / 16 in the address field
  const uint64_t qdesc0 = umma_smem_desc(smem_u32(sm.q), 128, 256);
  const uint64_t qmdesc0 = umma_smem_desc(smem_u32(sm.qm), 128, 256);
  constexpr uint64_t kQStep = C::kQBlk >> 4;
  for (int ii = i0; ii < i1; ++ii) {
    const Item it = p.items[ii];
    const int L = it.L, nst = item_stages<MODE>(it, L);
    for (int k0 = 0; k0 < nst;) {
      const int k1 = tc_tile_end<MODE>(it, L, k0, nst);
      const bool bf = tc_tile_bf16<MODE>(it, L, k0, k1);
      const int sb = tile % C::NS, su = tile / C::NS;
      if (su > 0) tc_wait(sm, &sm.s_empty[sb], (su - 1) & 1, p.status);
      const uint32_t d = tmem + C::colS + NH * sb;
      const int G = bf ? 9 : 10;
      uint64_t qdesc = qdesc0;  // query block (g, 0)
      for (int g = 0; g < G; ++g) {
        const int slot = g % C::NA;
        tc_wait(sm, &sm.a_full[slot], tc_get(a_use, slot) & 1, p.status);
        tc_fence_after();
        const uint32_t a = tmem + C::colA + C::kSlotCols * slot;
        if (g < 9) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) umma_f16_ts(d, a + 8 * kk, qdesc + kk * kQStep, idesc, g > 0 || kk > 0);
          if (!bf) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_f16_ts(d, a + 32 + 8 * kk, qdesc + kk * kQStep, idesc, true);
          }
        } else {
          umma_f16_ts(d, a, qmdesc0, idesc, true);
          umma_f16_ts(d, a + 8, qmdesc0 + kQStep, idesc, true);
        }
        umma_commit(&sm.a_empty[slot]);
        tc_bump(a_use, slot);
        qdesc += 4 * kQStep;
      }
      umma_commit(&sm.s_full[sb]);
      ++tile;
      k0 = k1;
    }
  }
}

// Aggregation issuer: per 16-token row group, one MMA per 128-channel block
// (O^T[c, h] += V^T[c, t] P^T[t, h]); an item's first MMA overwrites O^T once
// the previous item's epilogue has read it.
template <int MODE, int NH>
__device__ void tc_agg_issuer(const DecodeParams& p, TcSmem<NH>& sm, uint32_t tmem, int i0, int i1) {
  using C = TcCfg<NH>;
  constexpr uint32_t idesc = umma_idesc_f16(128, NH);
  int v_use = 0, tile = 0, item_n = 0;
  uint64_t ptdesc[C::NP];
#pragma unroll
  for (int k = 0; k < C::NP; ++k) ptdesc[k] = umma_smem_desc(smem_u32(sm.pt[k]), C::kPtLbo, C::kPtSbo);
  static_assert(C::kPtRg % 16 == 0, "P^T row groups on 16-byte boundaries");
  for (int ii = i0; ii < i1; ++ii, ++item_n) {
    const Item it = p.items[ii];
    const int L = it.L, nst = item_stages<MODE>(it, L);
    bool first = true;
    for (int k0 = 0; k0 < nst;) {
      const int k1 = tc_tile_end<MODE>(it, L, k0, nst);
      int nrg = 0;
      for (int k = k0; k < k1; ++k) nrg += item_stage<MODE>(it, L, k).kind == 1 ? 4 : 1;
      const int pb = tile % C::NP;
      tc_wait(sm, &sm.p_full[pb], (tile / C::NP) & 1, p.status);
      if (first && item_n > 0) tc_wait(sm, &sm.o_free, (item_n - 1) & 1, p.status);
      for (int j = 0; j < nrg; ++j) {
        const int vs = v_use % C::NV;
        tc_wait(sm, &sm.v_full[vs], (v_use / C::NV) & 1, p.status);
        tc_fence_after();
        const uint64_t bdesc = ptdesc[pb] + (uint64_t)(j * (C::kPtRg >> 4));
#pragma unroll
        for (int blk = 0; blk < 4; ++blk)
          umma_f16_ts(tmem + C::colO + NH * blk, tmem + C::colV + 32 * vs + 8 * blk, bdesc, idesc, !(first && j == 0));
        umma_commit(&sm.v_empty[vs]);
        ++v_use;
      }
      umma_commit(&sm.p_empty[pb]);
      first = false;
      ++tile;
      k0 = k1;
    }
  }
}

// ---------------------------------------------------------------------------
// Centered exact codes (q - 8 for 4-bit codes, q - 2 for 2-bit codes) as
// fp16 pairs: the same LOP3 + HFMA2 as the plain unpack with the center
// folded into the HFMA2's addend (1024 + m q scaled by 1/m, minus 1024/m +
// center). Centered operands keep the score accumulator near the size of
// the score itself (the plain codes add about mn * sum(Q) per group, which
// the min term takes back out, and fp32 rounding grows with that offset).
__device__ __forceinline__ uint32_t int4_pos_c(uint32_t w, uint32_t w8, int p) {
  switch (p) {
    case 0: return unpack_pair(w, 0x000F000Fu, kH1, 0xE408E408u);       // -1032
    case 1: return unpack_pair(w, 0x00F000F0u, kH1_16, 0xD480D480u);    // -72
    case 2: return unpack_pair(w8, 0x000F000Fu, kH1, 0xE408E408u);
    default: return unpack_pair(w8, 0x00F000F0u, kH1_16, 0xD480D480u);
  }
}
__device__ __forceinline__ uint32_t int2_pos_c(uint32_t w, uint32_t w8, int p) {
  const uint32_t x = p < 4 ? w : w8;
  switch (p & 3) {
    case 0: return unpack_pair(x, 0x00030003u, kH1, 0xE402E402u);      // -1026
    case 1: return unpack_pair(x, 0x000C000Cu, kH1_4, 0xDC08DC08u);    // -258
    case 2: return unpack_pair(x, 0x00300030u, kH1_16, 0xD420D420u);   // -66
    default: return unpack_pair(x, 0x00C000C0u, kH1_64, 0xCC80CC80u);  // -18
  }
}
template <int MODE>
__device__ __forceinline__ float tc_code_center(int g) { return (g < 8 && content_bits(MODE) == 2) ? 2.f : 8.f; }

// Score operand of one token row for group g (< 9): the (q - C) * s_hi and
// (q - C) * s_lo pairs (C the code center) of column pairs k = 16 HALF ..
// 16 HALF + 15 of the group (channels 2k, 2k + 1, natural order). Packed rows pass the group's code
// words (loaded once for both halves) and its (scale, min) meta word.
struct TcWords {
  uint32_t w[8];
};
template <int MODE>
__device__ __forceinline__ TcWords tc_load_words(const uint8_t* st, int prow, int g, int lane) {
  constexpr int CB = token_bytes(MODE);
  constexpr int CBITS = content_bits(MODE);
  constexpr int GBYTES = group_code_bytes(CBITS);
  TcWords t;
  const uint8_t* gp = st + prow * CB + (g < 8 ? g * GBYTES : 8 * GBYTES);
  if (g < 8 && CBITS == 2) {
    const uint4 wv = *reinterpret_cast<const uint4*>(gp);
    t.w[0] = wv.x; t.w[1] = wv.y; t.w[2] = wv.z; t.w[3] = wv.w;
    t.w[4] = t.w[5] = t.w[6] = t.w[7] = 0u;
  } else {
    // the two 16-byte halves in an order that alternates with bit 2 of the
    // lane: with 288- or 160-byte rows the eight lanes of a quarter warp then
    // read distinct banks
    const int hsel = (lane >> 2) & 1;
    const uint4 a = *reinterpret_cast<const uint4*>(gp + 16 * hsel);
    const uint4 b = *reinterpret_cast<const uint4*>(gp + 16 * (hsel ^ 1));
    const uint4 w0 = hsel ? b : a, w1 = hsel ? a : b;
    t.w[0] = w0.x; t.w[1] = w0.y; t.w[2] = w0.z; t.w[3] = w0.w;
    t.w[4] = w1.x; t.w[5] = w1.y; t.w[6] = w1.z; t.w[7] = w1.w;
  }
  return t;
}
template <int MODE, int HALF>
__device__ __forceinline__ void tc_row_half(const TcWords& t, uint32_t meta, const uint8_t* st, int kind, int prow,
                                            int g, bool want_lo, uint32_t (&hi)[16], uint32_t (&lo)[16]) {
  constexpr int CBITS = content_bits(MODE);
  if (MODE != MLAQ_BF16 && kind == 1) {
    const uint32_t sb = meta & 0xffffu, shb = sb & 0xfff0u;
    const __half s_hi = __ushort_as_half((unsigned short)shb);
    const __half s_lo = __hsub(__ushort_as_half((unsigned short)sb), s_hi);
    const __half2 SH = __half2half2(s_hi), SL = __half2half2(s_lo);
    if (g < 8 && CBITS == 2) {
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        const uint32_t w = t.w[wi], w8 = w >> 8;
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) {
          const int k = tc_col_int2(wi, pp);
          if ((k >> 4) != HALF) continue;
          const __half2 qv = u32_as_h2(int2_pos_c(w, w8, pp));
          hi[k & 15] = h2_as_u32(__hmul2(qv, SH));
          lo[k & 15] = h2_as_u32(__hmul2(qv, SL));
        }
      }
    } else {
#pragma unroll
      for (int wi = 0; wi < 8; ++wi) {
        const uint32_t w = t.w[wi], w8 = w >> 8;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int k = g < 8 ? tc_col_int4(wi, pp) : tc_col_rope(wi, pp);
          if ((k >> 4) != HALF) continue;
          const __half2 qv = u32_as_h2(int4_pos_c(w, w8, pp));
          hi[k & 15] = h2_as_u32(__hmul2(qv, SH));
          lo[k & 15] = h2_as_u32(__hmul2(qv, SL));
        }
      }
    }
  } else {
    // BF16 row (ring slot or BF16-mode page token): its value is the hi part
    const uint16_t* rp = reinterpret_cast<const uint16_t*>(st + prow * (kD * 2));
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const uint4 v = *reinterpret_cast<const uint4*>(rp + bf16_row_pos(kGroup * g + 8 * (4 * HALF + cc), prow));
      hi[4 * cc + 0] = bf2_to_h2(v.x);
      hi[4 * cc + 1] = bf2_to_h2(v.y);
      hi[4 * cc + 2] = bf2_to_h2(v.z);
      hi[4 * cc + 3] = bf2_to_h2(v.w);
    }
    if (want_lo) {
#pragma unroll
      for (int k = 0; k < 16; ++k) lo[k] = 0u;
    }
  }
}

// Query of sequence b, heads h0 .. h0 + NH - 1, into the score B operand
// (fp16; bf16 values convert exactly) and the min term's group sums (fp32
// sums split into fp16 hi + lo). Out-of-range values set MLAQ_DEV_RANGE.
template <int NH>
__device__ void tc_load_query(const DecodeParams& p, TcSmem<NH>& sm, int b, int h0, int tid, int nthreads) {
  using C = TcCfg<NH>;
  const uint16_t* ql = p.q_latent + ((size_t)b * p.H + h0) * kDL;
  const uint16_t* qr = p.q_rope + ((size_t)b * p.H + h0) * kDR;
  bool bad = false;
  for (int u = tid; u < NH * (kD / 8); u += nthreads) {
    const int h = u / (kD / 8), c8 = u % (kD / 8), c = 8 * c8;
    const uint4 v = c < kDL ? *reinterpret_cast<const uint4*>(ql + (size_t)h * kDL + c)
                            : *reinterpret_cast<const uint4*>(qr + (size_t)h * kDR + (c - kDL));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) bad |= (wv[e] & 0x7fffu) > 0x477fu || ((wv[e] >> 16) & 0x7fffu) > 0x477fu;
    const int g = c / kGroup, cg = c % kGroup;
    uint8_t* dst = sm.q + (4 * g + cg / 16) * C::kQBlk + (h >> 3) * 256 + ((cg % 16) >> 3) * 128 + (h & 7) * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(bf2_to_h2(v.x), bf2_to_h2(v.y), bf2_to_h2(v.z), bf2_to_h2(v.w));
  }
  named_bar_sync(2, 32 * C::kSW);  // the fp16 query is in shared memory
  for (int u = tid; u < NH * kGroups; u += nthreads) {
    const int h = u / kGroups, g = u % kGroups;
    float acc = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint4 v = *reinterpret_cast<const uint4*>(sm.q + (4 * g + c8 / 2) * C::kQBlk + (h >> 3) * 256 +
                                                      (c8 & 1) * 128 + (h & 7) * 16);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(u32_as_h2(wv[e]));
        acc += f.x + f.y;
      }
    }
    bad |= !(fabsf(acc) < 65520.f);
    const __half hi = __float2half_rn(acc);
    const __half lo = __float2half_rn(acc - __half2float(hi));
    // K elements 3g, 3g + 1, 3g + 2 of the 32: (hi, lo, hi)
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      const int e = 3 * g + t;
      *reinterpret_cast<__half*>(sm.qm + (e / 16) * C::kQBlk + (h >> 3) * 256 + ((e % 16) >> 3) * 128 + (h & 7) * 16 +
                                 (e % 8) * 2) = t == 1 ? lo : hi;
    }
  }
  if (bad) atomicOr(p.status, MLAQ_DEV_RANGE);
}

// Score warps: quadrant q = w % 4 (TMEM lanes 32q .. 32q + 31 = tile rows),
// half s = w / 4 (column half s of every group's operand and heads
// [s HPW, (s + 1) HPW) when there are two warps per quadrant).
template <int MODE, int NH>
__device__ void tc_score_warps(const DecodeParams& p, TcSmem<NH>& sm, uint32_t tmem, int i0, int i1, int w,
                               int lane) {
  using C = TcCfg<NH>;
  constexpr int HPW = C::HPW;
  const int q = w & 3, s = w >> 2;
  const int hoff = s * HPW;
  const int row = 32 * q + lane, rg = row >> 4, t16 = row & 15;
  const int h0 = blockIdx.x * NH;
  const int H = p.H;
  int gs = 0, tile = 0, item_n = 0, cur_b = -1;
  int a_use[C::NAS];
#pragma unroll
  for (int k = 0; k < C::NAS; ++k) a_use[k] = 0;
  // the min term's padding columns (K 18 .. 31) stay zero
  for (int u = threadIdx.x; u < 2 * C::kQBlk / 16; u += 32 * C::kSW)
    reinterpret_cast<uint4*>(sm.qm)[u] = make_uint4(0u, 0u, 0u, 0u);
  float l_part[HPW];
  for (int ii = i0; ii < i1; ++ii, ++item_n) {
    const Item it = p.items[ii];
    const int L = it.L, nst = item_stages<MODE>(it, L);
    const bool single = p.item_start[it.b + 1] - p.item_start[it.b] == 1;
    if (it.b != cur_b) {
      cur_b = it.b;
      tc_load_query<NH>(p, sm, it.b, h0, threadIdx.x, 32 * C::kSW);
      fence_view_async_shared();
    }
    if (lane == 0 && q == 0)
      for (int h = 0; h < HPW; ++h) sm.m_run[hoff + h] = -INFINITY;
#pragma unroll
    for (int h = 0; h < HPW; ++h) l_part[h] = 0.f;
    named_bar_sync(2, 32 * C::kSW);  // query and running max in place
    for (int k0 = 0; k0 < nst;) {
      const int k1 = tc_tile_end<MODE>(it, L, k0, nst);
      const int nstg = k1 - k0;
      for (int k = 0; k < nstg; ++k) tc_wait(sm, &sm.full[(gs + k) % C::NSTG], ((gs + k) / C::NSTG) & 1, p.status);
      // this row's stage
      int si = 0, base = 0, nrg = 0;
      StageRef sref = item_stage<MODE>(it, L, k0);
      for (int k = 0; k < nstg; ++k) {
        const StageRef st_k = item_stage<MODE>(it, L, k0 + k);
        const int cnt = st_k.kind == 1 ? 4 : 1;
        if (rg >= nrg) {
          si = k;
          base = nrg;
          sref = st_k;
        }
        nrg += cnt;
      }
      const bool in_tile = rg < nrg;
      const int sub = in_tile ? rg - base : 0;
      const int prow = sref.kind == 1 ? 16 * sub + t16 : t16;
      const int buf = (gs + si) % C::NSTG;
      const uint8_t* st = sm.stage[buf];
      const bool valid = in_tile && !sm.stage_bad[buf] && row_valid<MODE>(sref, prow, L);
      const bool bf = tc_tile_bf16<MODE>(it, L, k0, k1);
      const int G = bf ? 9 : 10;
      // ---- score operands: every group is written by the 4 SWQ warps; with
      // two warps per quadrant, warp s writes column half s. The operand is
      // built in registers before waiting for its slot, so the unpack overlaps
      // the MMAs still reading the slot.
      for (int g = 0; g < G; ++g) {
        const int slot = g % C::NA;
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + C::colA + C::kSlotCols * slot;
        if (g < 9) {
          TcWords wds;
          uint32_t meta = 0u;
          if (MODE != MLAQ_BF16 && sref.kind == 1) {
            wds = tc_load_words<MODE>(st, prow, g, lane);
            meta = *reinterpret_cast<const uint32_t*>(st + page_code_bytes(MODE) + prow * kMetaTok + 4 * g);
          }
          if constexpr (C::SWQ == 2) {
            uint32_t hi[16], lo[16];
            if (s == 0)
              tc_row_half<MODE, 0>(wds, meta, st, sref.kind, prow, g, !bf, hi, lo);
            else
              tc_row_half<MODE, 1>(wds, meta, st, sref.kind, prow, g, !bf, hi, lo);
            const int use = tc_get(a_use, slot);
            if (use > 0) tc_wait(sm, &sm.a_empty[slot], (use - 1) & 1, p.status);
            tc_fence_after();
            tmem_st_32x32b_x16(ta + 16 * s, hi);
            if (!bf) tmem_st_32x32b_x16(ta + 32 + 16 * s, lo);
          } else {
            uint32_t hi0[16], lo0[16], hi1[16], lo1[16];
            tc_row_half<MODE, 0>(wds, meta, st, sref.kind, prow, g, !bf, hi0, lo0);
            tc_row_half<MODE, 1>(wds, meta, st, sref.kind, prow, g, !bf, hi1, lo1);
            const int use = tc_get(a_use, slot);
            if (use > 0) tc_wait(sm, &sm.a_empty[slot], (use - 1) & 1, p.status);
            tc_fence_after();
            tmem_st_32x32b_x16(ta, hi0);
            tmem_st_32x32b_x16(ta + 16, hi1);
            if (!bf) {
              tmem_st_32x32b_x16(ta + 32, lo0);
              tmem_st_32x32b_x16(ta + 48, lo1);
            }
          }
        } else {
          // midpoint term (written by half 0): the group midpoints d_j = mn_j
          // + C s_j (exact in fp32) split into fp16 hi + lo; K elements 3j,
          // 3j + 1, 3j + 2 hold (d_hi, d_hi, d_lo) against (sum_hi, sum_lo,
          // sum_hi) of the query
          uint32_t mv[16];
          if (s == 0) {
            __half dh[9], dl[9];
#pragma unroll
            for (int j = 0; j < 9; ++j) {
              dh[j] = __ushort_as_half(0);
              dl[j] = __ushort_as_half(0);
            }
            if (MODE != MLAQ_BF16 && sref.kind == 1) {
#pragma unroll
              for (int j = 0; j < 9; ++j) {
                const uint32_t mt =
                    *reinterpret_cast<const uint32_t*>(st + page_code_bytes(MODE) + prow * kMetaTok + 4 * j);
                const float2 sm2 = __half22float2(u32_as_h2(mt));  // (s, mn)
                const float d = __fmaf_rn(tc_code_center<MODE>(j), sm2.x, sm2.y);
                dh[j] = __float2half_rn(d);
                dl[j] = __float2half_rn(d - __half2float(dh[j]));
              }
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              __half e2[2];
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const int e = 2 * c + t;
                e2[t] = e < 27 ? ((e % 3) < 2 ? dh[e / 3] : dl[e / 3]) : __ushort_as_half(0);
              }
              mv[c] = h2_as_u32(__halves2half2(e2[0], e2[1]));
            }
          }
          const int use = tc_get(a_use, slot);
          if (use > 0) tc_wait(sm, &sm.a_empty[slot], (use - 1) & 1, p.status);
          tc_fence_after();
          if (s == 0) tmem_st_32x32b_x16(ta, mv);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.a_full[slot]);
        tc_bump(a_use, slot);
      }
      // the tile's stages are no longer read by this warp
      __syncwarp();
      if (lane == 0)
        for (int k = 0; k < nstg; ++k) mbar_arrive(&sm.empty[(gs + k) % C::NSTG]);
      gs += nstg;
      // ---- scores of this row for the warp's heads
      const int sb = tile % C::NS;
      tc_wait(sm, &sm.s_full[sb], (tile / C::NS) & 1, p.status);
      tc_fence_after();
      uint32_t sv[HPW];
      {
        const uint32_t ts = tmem + ((uint32_t)(32 * q) << 16) + C::colS + NH * sb + hoff;
        if constexpr (HPW == 32)
          tmem_ld_32x32b_x32(ts, sv);
        else
          tmem_ld_32x32b_x16(ts, sv);
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_empty[sb]);
      // ---- online softmax: one token row, HPW heads; the running max is
      // shared by the CTA (lazy: raised only when a score exceeds it by 2^14)
      float x[HPW];
      int tok = 0;
      if (p.q_len > 1 && valid) tok = row_token<MODE>(sref, prow, L);
      bool need = false;
#pragma unroll
      for (int h = 0; h < HPW; ++h) {
        bool ok = valid;
        if (p.q_len > 1) ok = ok && tok < L - (p.q_len - 1 - (h0 + hoff + h) / p.h_per_q);
        x[h] = ok ? __uint_as_float(sv[h]) * p.scale_log2 : -INFINITY;
        need |= x[h] > sm.m_run[hoff + h] + 14.f;
      }
      const int par = tile & 1;
      const bool wneed = __any_sync(0xffffffffu, need);
      if (lane == 0) sm.vote[par][w] = wneed;
      // the P^T buffer (and its alpha) are free once the aggregation of the
      // tile that used them last completed
      const int pb = tile % C::NP, pu = tile / C::NP;
      if (pu > 0) tc_wait(sm, &sm.p_empty[pb], (pu - 1) & 1, p.status);
      named_bar_sync(2, 32 * C::kSW);
      bool any = false;
#pragma unroll
      for (int k = 0; k < C::kSW; ++k) any |= sm.vote[par][k] != 0;
      bool rs = false;
      if (any) {  // rare after an item's first tile: the tile max of every head
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          float v = x[h];
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
          if (lane == h) sm.red[par][q][hoff + h] = v;
        }
        named_bar_sync(2, 32 * C::kSW);
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          const float tmax = fmaxf(fmaxf(sm.red[par][0][hoff + h], sm.red[par][1][hoff + h]),
                                   fmaxf(sm.red[par][2][hoff + h], sm.red[par][3][hoff + h]));
          const float m_old = sm.m_run[hoff + h];
          const bool upd = tmax > m_old + 14.f;  // m_old = -inf gives alpha = 0
          const float alpha = upd ? ex2(m_old - tmax) : 1.f;
          l_part[h] *= alpha;
          rs |= upd;
          if (q == 0 && lane == h) sm.alpha[pb][hoff + h] = alpha;
        }
        named_bar_sync(2, 32 * C::kSW);  // every warp read the old running max
        if (q == 0 && lane < HPW) {
          const int hh = hoff + lane;
          const float tmax = fmaxf(fmaxf(sm.red[par][0][hh], sm.red[par][1][hh]),
                                   fmaxf(sm.red[par][2][hh], sm.red[par][3][hh]));
          if (tmax > sm.m_run[hh] + 14.f) sm.m_run[hh] = tmax;
        }
        named_bar_sync(2, 32 * C::kSW);  // the new running max is in place
      }
#pragma unroll
      for (int h = 0; h < HPW; ++h) {
        const float m = sm.m_run[hoff + h];
        const float mref = m == -INFINITY ? 0.f : m;  // nothing valid yet: p = 0
        x[h] = ex2(x[h] - mref);
        l_part[h] += x[h];
      }
      // ---- P^T for the aggregation, the rescale flag for the value warps
      if (q == 0 && lane == 0) sm.rs_flag[pb][s] = rs;
      if (in_tile) {
        uint8_t* pt = sm.pt[pb] + rg * C::kPtRg;
        const int K = tc_kpos(t16);
        const int koff = (K >> 3) * C::kPtLbo + (K & 7) * 2;
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          const int hh = hoff + h;
          *reinterpret_cast<__half*>(pt + (hh >> 3) * C::kPtSbo + (hh & 7) * 16 + koff) = __float2half_rn(x[h]);
        }
      }
      fence_view_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[pb]);
      ++tile;
      k0 = k1;
    }
    // ---- item end: l over the tile rows, lse, and (l, m) for the value warps
    const int ip = item_n & 1;
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
      float v = l_part[h];
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == h) sm.red[0][q][hoff + h] = v;  // red[0] is free: the tiles' reductions are done
    }
    named_bar_sync(2, 32 * C::kSW);
    if (q == 0 && lane < HPW) {
      const int hh = hoff + lane;
      const float l = sm.red[0][0][hh] + sm.red[0][1][hh] + sm.red[0][2][hh] + sm.red[0][3][hh];
      const float m = sm.m_run[hh];
      sm.fin_l[ip][hh] = l;
      sm.fin_m[ip][hh] = m;
      const float lse_v = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (single)
        p.lse[(size_t)it.b * H + h0 + hh] = lse_v;
      else
        p.lse_part[(size_t)ii * H + h0 + hh] = lse_v;
    }
    named_bar_sync(1, 32 * (C::kSW + 4));  // (l, m) of the item are in shared memory
  }
}

// Value fragments of a 16-row group: content groups 2q, 2q + 1 (channels
// 128q .. 128q + 127) of rows lr, lr + 8, dequantized to fp16 and transposed
// for the V^T store (vv[kk & 1][4 blk + e], blk = 2j + kk / 2).
template <int MODE>
__device__ __forceinline__ void tc_value_fragments(const uint8_t* st, const StageRef& sref, int sub, bool live, int L,
                                                   int q, int r, int i, uint32_t (&vv)[2][16]) {
  constexpr int CB = token_bytes(MODE);
  constexpr int CBITS = content_bits(MODE);
  constexpr int GBYTES = group_code_bytes(CBITS);
  uint32_t ch[2][4][4];
  if (MODE != MLAQ_BF16 && sref.kind == 1) {
    const int lr = 16 * sub + r;
    const bool v0 = live && row_valid<MODE>(sref, lr, L);
    const bool v1 = live && row_valid<MODE>(sref, lr + 8, L);
    const uint8_t* mtab = st + page_code_bytes(MODE);
    uint32_t mx[2], my[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int gg = 2 * q + j;
      const uint32_t mxr = *reinterpret_cast<const uint32_t*>(mtab + lr * kMetaTok + 4 * gg);
      const uint32_t myr = *reinterpret_cast<const uint32_t*>(mtab + (lr + 8) * kMetaTok + 4 * gg);
      mx[j] = v0 ? mxr : 0u;
      my[j] = v1 ? myr : 0u;
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
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const __half2 s2x = __low2half2(u32_as_h2(mx[j])), m2x = __high2half2(u32_as_h2(mx[j]));
      const __half2 s2y = __low2half2(u32_as_h2(my[j])), m2y = __high2half2(u32_as_h2(my[j]));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t* v = &vv[kk & 1][4 * (2 * j + (kk >> 1))];
        v[0] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][0]), s2x, m2x)));
        v[1] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][1]), s2y, m2y)));
        v[2] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][2]), s2x, m2x)));
        v[3] = movmatrix_t(h2_as_u32(__hfma2(u32_as_h2(ch[j][kk][3]), s2y, m2y)));
      }
    }
  } else {
    // BF16 rows (ring chunk or BF16 page quarter): rows r, r + 8 of the stage
    const bool v0 = live && row_valid<MODE>(sref, r, L);
    const bool v1 = live && row_valid<MODE>(sref, r + 8, L);
    const uint16_t* rx = reinterpret_cast<const uint16_t*>(st + r * (kD * 2));
    const uint16_t* ry = reinterpret_cast<const uint16_t*>(st + (r + 8) * (kD * 2));
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int c = 64 * (2 * q + j) + 16 * kk + 2 * i;
        const int e0 = bf16_row_pos(c, r), e1 = bf16_row_pos(c + 8, r);
        uint32_t* v = &vv[kk & 1][4 * (2 * j + (kk >> 1))];
        v[0] = movmatrix_t(v0 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(rx + e0)) : 0u);
        v[1] = movmatrix_t(v1 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(ry + e0)) : 0u);
        v[2] = movmatrix_t(v0 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(rx + e1)) : 0u);
        v[3] = movmatrix_t(v1 ? bf2_to_h2(*reinterpret_cast<const uint32_t*>(ry + e1)) : 0u);
      }
  }
}

// Value warps: quadrant q (V^T and O^T lanes 32q .. 32q + 31, content
// channels 128q .. 128q + 127).
template <int MODE, int NH>
__device__ void tc_value_warps(const DecodeParams& p, TcSmem<NH>& sm, uint32_t tmem, int i0, int i1, int q,
                               int lane) {
  using C = TcCfg<NH>;
  const int r = lane >> 2, i = lane & 3;
  const int h0 = blockIdx.x * NH;
  const int H = p.H;
  int gs = 0, v_use = 0, tile = 0, item_n = 0;
  for (int ii = i0; ii < i1; ++ii, ++item_n) {
    const Item it = p.items[ii];
    const int L = it.L, nst = item_stages<MODE>(it, L);
    const bool single = p.item_start[it.b + 1] - p.item_start[it.b] == 1;
    bool first = true;
    for (int k0 = 0; k0 < nst;) {
      const int k1 = tc_tile_end<MODE>(it, L, k0, nst);
      const int nstg = k1 - k0;
      for (int k = 0; k < nstg; ++k) tc_wait(sm, &sm.full[(gs + k) % C::NSTG], ((gs + k) / C::NSTG) & 1, p.status);
      const int pb = tile % C::NP;
      int j = 0;
      for (int k = 0; k < nstg; ++k) {
        const StageRef sref = item_stage<MODE>(it, L, k0 + k);
        const int buf = (gs + k) % C::NSTG;
        const uint8_t* st = sm.stage[buf];
        const bool live = !sm.stage_bad[buf];
        const int nsub = sref.kind == 1 ? 4 : 1;
        for (int sub = 0; sub < nsub; ++sub, ++j) {
          uint32_t vv[2][16];
          tc_value_fragments<MODE>(st, sref, sub, live, L, q, r, i, vv);
          if (j == 0) {
            // the softmax of this tile may have raised the running max: scale
            // O^T first (after the previous tile's aggregation completed)
            tc_wait(sm, &sm.p_full[pb], (tile / C::NP) & 1, p.status);
            if (!first && (sm.rs_flag[pb][0] | (C::SWQ == 2 ? sm.rs_flag[pb][1] : 0))) {
              const int pt = tile - 1;
              tc_wait(sm, &sm.p_empty[pt % C::NP], (pt / C::NP) & 1, p.status);
              tc_fence_after();
#pragma unroll 1
              for (int blk = 0; blk < 4; ++blk)
#pragma unroll 1
                for (int hc = 0; hc < NH / 16; ++hc) {
                  uint32_t v[16];
                  const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + C::colO + NH * blk + 16 * hc;
                  tmem_ld_32x32b_x16(ta, v);
                  tmem_wait_ld();
#pragma unroll
                  for (int h = 0; h < 16; ++h) {
                    const int hh = 16 * hc + h;
                    const float a = sm.rs_flag[pb][C::SWQ == 2 ? hh / C::HPW : 0] ? sm.alpha[pb][hh] : 1.f;
                    v[h] = __float_as_uint(__uint_as_float(v[h]) * a);
                  }
                  tmem_st_32x32b_x16(ta, v);
                }
              tmem_wait_st();
            }
          }
          const int vs = v_use % C::NV;
          if (v_use >= C::NV) tc_wait(sm, &sm.v_empty[vs], ((v_use / C::NV) - 1) & 1, p.status);
          tc_fence_after();
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2)
            tmem_st_16x256b_x4(tmem + ((uint32_t)(32 * q + 16 * k2) << 16) + C::colV + 32 * vs, vv[k2]);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.v_full[vs]);
          ++v_use;
        }
      }
      __syncwarp();
      if (lane == 0)
        for (int k = 0; k < nstg; ++k) mbar_arrive(&sm.empty[(gs + k) % C::NSTG]);
      gs += nstg;
      first = false;
      ++tile;
      k0 = k1;
    }
    // ---- epilogue: O^T / l, bf16 out (single item) or fp16 partial
    named_bar_sync(1, 32 * (C::kSW + 4));
    {
      const int lt = tile - 1;
      tc_wait(sm, &sm.p_empty[lt % C::NP], (lt / C::NP) & 1, p.status);  // the item's last MMAs completed
    }
    tc_fence_after();
    const int ip = item_n & 1;
    __half* op = p.o_part + ((size_t)ii * H + h0) * kDL;
#pragma unroll 1
    for (int hc = 0; hc < NH / 16; ++hc) {
      float inv[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float l = sm.fin_l[ip][16 * hc + h];
        inv[h] = l > 0.f ? 1.f / l : 0.f;
      }
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tmem + ((uint32_t)(32 * q) << 16) + C::colO + NH * blk + 16 * hc, v);
        tmem_wait_ld();
        const int c = 128 * q + 64 * (blk >> 1) + 16 * (2 * (blk & 1) + (lane >> 4)) + (lane & 15);
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const int hq = 16 * hc + h;
          const float val = inv[h] != 0.f ? __uint_as_float(v[h]) * inv[h] : 0.f;
          if (single)
            p.out[((size_t)it.b * H + h0 + hq) * kDL + c] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
          else
            op[(size_t)hq * kDL + c] = __float2half_rn(val);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.o_free);
  }
}

template <int MODE, int NH>
__global__ void __launch_bounds__(TcCfg<NH>::kThreads, 1) decode_tc_kernel(DecodeParams p) {
  using C = TcCfg<NH>;
  using SM = TcSmem<NH>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int cta = blockIdx.y;
  pdl_wait();  // the plan
  pdl_launch_dependents();
  const int i0 = p.cta_item_start[cta], i1 = p.cta_item_start[cta + 1];
  if (i0 >= i1) return;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int k = 0; k < C::NSTG; ++k) {
      mbar_init(&sm.full[k], 1);
      mbar_init(&sm.empty[k], C::kSW + 4);
    }
    for (int k = 0; k < C::NAS; ++k) {
      mbar_init(&sm.a_full[k], C::kSW);
      mbar_init(&sm.a_empty[k], 1);
    }
    for (int k = 0; k < C::NS; ++k) {
      mbar_init(&sm.s_full[k], 1);
      mbar_init(&sm.s_empty[k], C::kSW);
    }
    for (int k = 0; k < C::NV; ++k) {
      mbar_init(&sm.v_full[k], 4);
      mbar_init(&sm.v_empty[k], 1);
    }
    for (int k = 0; k < C::NP; ++k) {
      mbar_init(&sm.p_full[k], C::kSW);
      mbar_init(&sm.p_empty[k], 1);
    }
    mbar_init(&sm.o_free, 4);
    sm.abort = 0;
    fence_mbar_init();
    fence_proxy_async();
  }
  if (w == 0) {
    tmem_alloc(&sm.tmem_base, C::kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (w < C::kSW) {
    tc_score_warps<MODE, NH>(p, sm, tmem, i0, i1, w, lane);
  } else if (w < C::kSW + 4) {
    tc_value_warps<MODE, NH>(p, sm, tmem, i0, i1, w - C::kSW, lane);
  } else if (w == C::wProd) {
    if (lane == 0) tc_producer<MODE, NH>(p, sm, cta, i0, i1);
  } else if (w == C::wSIss) {
    if (lane == 0) tc_score_issuer<MODE, NH>(p, sm, tmem, i0, i1);
  } else {
    if (lane == 0) tc_agg_issuer<MODE, NH>(p, sm, tmem, i0, i1);
  }
  // every MMA completed: the value warps waited for the last aggregation
  // commit, the score warps for the last score commit
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (w == 0) tmem_dealloc(tmem, C::kCols);
}

}  // namespace mlaq
