// kvq_decode_tc.cu -- split-KV decode attention on the tensor cores (head_dim
// 128, up to 4 query heads per KV head, INT4, INT3 or INT2 codes).
//
// What it computes is the same as the generic kernel: O = softmax(q K^T /
// sqrt(d)) V over the packed tokens (dequantized min + code * scale, InnerQ page
// section 3.1) and the fp16 residual window (BitDecoding page section 2.2), all
// query heads of one KV head served by one read of the cache (BitDecoding page
// section 2.3).  How:
//
//  * 128-token tiles (192 for long INT2 splits in a grid of one wave) -- K
//    codes, V codes (2D TMA tile loads), K params, V params
//    (1D bulk copies: a tile's params are 2 KB of contiguous 16-byte rows, which
//    a tile load would move row by row) -- stream into a 2-stage shared-memory
//    ring guarded by mbarriers (the asynchronous staging of the BitDecoding page,
//    section 2.3, done with the bulk tensor copy instead of per-thread
//    cp.async).  One thread issues the first stages up front; the warp that
//    releases a stage last refills it at once.  Code
//    tiles use the TMA 64-byte (INT4) or 32-byte (INT2) swizzle, the XOR
//    swizzle of the BitDecoding page's equation (2), which makes every ldmatrix
//    below conflict-free.
//  * Four warps take 32 tokens (two independent 16-token sub-tiles) each per
//    tile (48 tokens, three sub-tiles, in the 192-token variant).  ldmatrix
//    brings code words to registers, and a single AND turns
//    two codes into one exact half2: a code c sitting in the low mantissa bits
//    of an fp16 whose exponent field is zero is the subnormal c * 2^-24 (a code
//    at bit offset 2 or 4 is 4c or 16c times 2^-24).  The tensor cores take
//    these exact operands as they are; the per-position weight 1/4/16 is
//    divided out of the q operand (K side) or out of the output row (V side),
//    and 2^24 goes into the softmax scale.  Scale and min are applied in fp32.
//  * QK:  S^T = K q^T with tokens on M (mma.sync m16n8k16, fp32 accumulate).
//    Two groups share one MMA through a block-diagonal q operand (column
//    2 * query + group bit), so each thread holds one query for both groups,
//    then  s = sum_g scale_g * acc_g + min_g * sum_{d in g} q_d.
//  * Online softmax in fp32 (exp2 domain) with a lazy rescale: the running max
//    only moves when it grows by more than 2^8, and the warp reduces it only
//    when one of a thread's own rows lies that far above it.
//  * PV:  O^T = c^T (p * scale)^T with V codes read through ldmatrix.trans.
//    Another MMA accumulates sum p * min_g and sum p (= l), so O = O_c +
//    sum_g p min_g.  p and p * scale enter as two fp16 parts (the rounded value
//    and the rest): one fp16 part alone would carry 11 bits, and an output of
//    magnitude 8 then moves by up to 2e-3 when one token holds most of the
//    weight.  INT4 (and INT3): each code MMA takes the rows of one group and
//    spends its 8 columns on 4 queries x the 2 parts.  INT2: a group spans half
//    of the lanes' code units, so its MMAs serve two groups through the columns
//    (2 * query + group bit), each part in an MMA of its own.
//  * The fp16 tokens -- the residual window, then the attention-sink rows
//    (InnerQ page section 2.3) -- get splits of their own, 64 rows each (all
//    loads of a split in one round, tensor cores), so no packed split waits on
//    them.  In a grid of several waves the last packed split of each
//    (sequence, KV head) takes them instead, once its stage ring is idle.
//  * Per-warp states merge in shared memory.  The first split of a KV head to
//    finish its first tile sets the head's reference max per query (atomicCAS);
//    every split adds its (o, l), scaled to that reference, into the head's fp32
//    accumulators (vector red.add), and the last split to finish divides by l.
//    A split whose max lies too far above the reference sends the head to the
//    exact log-sum-exp merge of the split partials (combine_unit) instead.  A
//    head with a single split writes its output straight from its own state.
//  * Three CTAs per SM (168 registers each) for grids of one wave: twelve warps
//    hide the latency of the dequantize-and-MMA chain; four (128 registers) for
//    grids of several waves.
//  * 3-bit codes (TurboQuant page section 3.1) arrive as plain 48-byte rows;
//    each warp widens its 32 rows to INT4 nibbles in a buffer of its own (the
//    INT4 swizzle), and the INT4 arithmetic runs on that buffer.
//  * Paged caches (32-token pages through a block table, TurboQuant page
//    section 6.1): packed splits start on page boundaries and a stage is filled
//    by one 32-row tile load per page of the pool instead of one 128-row load.
//
// Every mbarrier wait is bounded; a wait that runs out sets KVQ_ERRBIT_TIMEOUT.
#include <math.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "kvq_decode_common.cuh"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int D = 128;
constexpr int NG = D / kGroup;  // 4 groups per row
constexpr int QB = 4;           // query heads per CTA
constexpr int NCW = 4;          // warps; each takes a quarter of every tile
constexpr int NTHREADS = NCW * 32;
// CTAs per SM (CPS, a template parameter): 3 (12 warps, up to 168 registers,
// ~47 KB of shared memory each) for grids of one wave; 4 (16 warps, 128
// registers) for grids of several waves, where more warps hide more latency
// and the ramp of each CTA is overlapped by the others.
static_assert(NCW == QB, "the merge gives each warp one query");

// TT, tokens per pipeline stage: 128 (two independent 16-token sub-tiles per
// warp), or 192 (three) for INT2 splits of many tiles in a grid of one wave --
// the third sub-tile hides more of each warp's latency chain, which pays once a
// split is long enough that its larger first tile and ragged last one do not
// matter (contiguous caches only: a warp's 48 rows would straddle pages).
template <int BITS, int CPS, int TT>
struct Geo {
  static constexpr int T = TT;
  static constexpr int NSUB = TT / (16 * NCW);  // sub-tiles per warp per stage
  static constexpr int WR = 16 * NSUB;          // a warp's rows of the stage
  static_assert(TT == 128 || TT == 192, "two or three sub-tiles per warp");
  static constexpr int CB = BITS == 3 ? 4 : BITS;  // code width of the arithmetic
  static constexpr int RB = D * BITS / 8;      // code bytes per token row
  static constexpr int CODE_TILE = T * RB;     // 8192 (INT4) / 4096 (INT2) at 128 tokens
  static constexpr int PAR_TILE = T * NG * 4;  // 2048 at 128 tokens
  static constexpr int KC = 0;
  static constexpr int VC = CODE_TILE;
  static constexpr int KP = 2 * CODE_TILE;
  static constexpr int VP = 2 * CODE_TILE + PAR_TILE;
  static constexpr int STAGE = 2 * CODE_TILE + 2 * PAR_TILE;  // 20 KB / 12 KB
  // One tile in flight while the other is read: 20 KB (INT4) / 16 KB (INT3) /
  // 12 KB (INT2) of copies per CTA ahead of the compute.  Deeper rings (3 INT4
  // or 5 INT2 stages at 3 CTAs per SM, 4 INT2 at 4) were slower or no faster:
  // a tile's compute outlasts a copy's latency, and the extra bytes in flight
  // only delay the other CTAs' tiles.
  static constexpr int NSTAGE = 2;
  // INT3: per warp its widened rows of K and of V, 64 bytes each
  static constexpr int XBUF = BITS == 3 ? NCW * 2 * WR * 64 : 0;
  static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned");
};

// Shared scratch for the final merge (overlaps the stage ring once it is idle).
struct MergeSmem {
  float o[NCW][QB][D];
  float m[NCW][QB];
  float l[NCW][QB];
  float mn[NCW][9][8];
};

// The merge scratch, then the fused step's extra tokens [2][2][D] fp32, then a
// residual split's K and V rows overlap the stage ring (residual splits never
// use the ring; packed splits reuse it for the merge once it is idle).
constexpr size_t kResTilesOff = (sizeof(MergeSmem) + 4 * D * sizeof(float) + 127) & ~(size_t)127;
template <int BITS, int CPS, int TT>
constexpr size_t tc_smem_bytes() {
  using G = Geo<BITS, CPS, TT>;
  constexpr size_t ring = (size_t)G::NSTAGE * G::STAGE + G::XBUF;
  constexpr size_t res = kResTilesOff + 2 * 64 * (2 * D + 16);  // kResRows rows of K and V
  return 1024 + (ring > res ? ring : res);
}

// ------------------------------------------------------- code conversion ---

// One 3-bit code row (128 codes, 48 bytes, code e at bits 3e) widened to INT4
// (64 bytes, code e at bits 4e), stored as row `lrow` of a 32-row INT4 buffer
// at `dst` with the INT4 tile swizzle (16-byte chunk ^= (lrow >> 1) & 3).  Each
// output word takes 24 source bits (eight codes) and spreads them to nibbles in
// three mask-and-shift steps: 12-bit halves to 16-bit halves, 6-bit pairs to
// bytes, 3-bit codes to nibbles.
__device__ __forceinline__ void widen_row3(const uint8_t* src, uint32_t dst, int lrow) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  const uint4 a = s4[0], b = s4[1], c = s4[2];
  const uint32_t w[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {  // one 16-byte chunk = one group of 32 codes
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int bit = 24 * (4 * ch + k);
      const int wi = bit >> 5, sh = bit & 31;
      uint32_t x = w[wi] >> sh;
      if (sh > 8) x |= w[wi + 1] << (32 - sh);  // the 24 bits straddle two words
      x &= 0xFFFFFFu;
      uint32_t y = (x & 0xFFFu) | ((x & 0xFFF000u) << 4);
      y = (y & 0x003F003Fu) | ((y & 0x0FC00FC0u) << 2);
      o[k] = (y & 0x07070707u) | ((y & 0x38383838u) << 1);
    }
    const uint32_t addr = dst + lrow * 64 + ((ch ^ ((lrow >> 1) & 3)) << 4);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o[0]), "r"(o[1]),
                 "r"(o[2]), "r"(o[3])
                 : "memory");
  }
}

// Code words -> exact half2 operands (subnormal fp16, see the file comment).
// INT4: nibble j of each 16-bit half (j = 0..3) -> out[j] = (nibble j of the
// low half, nibble j of the high half) times W4[j] * 2^-24.
__device__ __forceinline__ void split_int4(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  o[0] = w & 0x000F000Fu;
  o[1] = w & 0x00F000F0u;
  o[2] = w8 & 0x000F000Fu;
  o[3] = w8 & 0x00F000F0u;
}
__host__ __device__ constexpr float w4_weight(int j) { return (j & 1) ? 16.f : 1.f; }

// INT2: code j of each 16-bit half (bits 2j, 2j+1; j = 0..7) -> out[j] = (code
// j of the low half, code j of the high half) times W2[j] * 2^-24, W2 = 1, 4,
// 16, 1, 4, 16, 1, 4 (shifts by 6 and 12 keep every weight <= 16).
__device__ __forceinline__ void split_int2(uint32_t w, uint32_t (&o)[8]) {
  const uint32_t w6 = w >> 6, w12 = w >> 12;
  o[0] = w & 0x00030003u;
  o[1] = w & 0x000C000Cu;
  o[2] = w & 0x00300030u;
  o[3] = w6 & 0x00030003u;
  o[4] = w6 & 0x000C000Cu;
  o[5] = w6 & 0x00300030u;
  o[6] = w12 & 0x00030003u;
  o[7] = w12 & 0x000C000Cu;
}
__host__ __device__ constexpr float w2_weight(int j) {
  return (j % 3) == 0 ? 1.f : ((j % 3) == 1 ? 4.f : 16.f);
}

constexpr float kTwo24 = 16777216.f;  // 2^24
constexpr int kPagePrefetch = 64;     // page ids of a split kept in shared memory
// A split whose max (log2 units) is more than this above the head's reference
// could overflow fp32 once scaled to it: the head then takes the exact merge.
constexpr float kRefSlack = 80.f;

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// QK of one 16-token sub-tile (rows r0 .. r0+15 of the stage): acc[P] holds the
// per-pair partial dot products (fragment layout of S^T = K q^T), times 2^-24.
// A operand registers: a0 = (row g, k 2t..2t+1), a1 = (row g+8, same k),
// a2 = (row g, k 2t+8..2t+9), a3 = (row g+8, same k); one k-step uses one code
// position, so one weight, which the matching bq fragment has divided out.
template <int BITS>
__device__ __forceinline__ void qk_subtile(uint32_t kc, int r0, int lane,
                                           const uint32_t (&bq)[2][4][2], float (&acc)[2][4]) {
  const int mj = lane >> 3, mi = lane & 7;
  const int lrow = r0 + (mj & 1) * 8 + mi;
#pragma unroll
  for (int P = 0; P < 2; ++P)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[P][r] = 0.f;
  if (BITS == 4) {
#pragma unroll
    for (int P = 0; P < 2; ++P) {
      // w0/w1: rows g/g+8, group P; w2/w3: the same rows, group P+2 (dims 8t..8t+7)
      const int chunk = (mj < 2) ? P : P + 2;
      const uint32_t addr = kc + lrow * 64 + ((chunk ^ ((lrow >> 1) & 3)) << 4);
      uint32_t w0, w1, w2, w3;
      ptx::ldmatrix_x4(addr, w0, w1, w2, w3);
      uint32_t c0[4], c1[4], c2[4], c3[4];
      split_int4(w0, c0);
      split_int4(w1, c1);
      split_int4(w2, c2);
      split_int4(w3, c3);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        ptx::mma_16816(acc[P], c0[k], c1[k], c2[k], c3[k], bq[P][k][0], bq[P][k][1]);
    }
  } else {
    // w[2P]/w[2P+1]: rows g/g+8, dims 64P + 16t .. +15 (one group per thread)
    const int chunk = mj >> 1;
    const uint32_t addr = kc + lrow * 32 + ((chunk ^ ((lrow >> 2) & 1)) << 4);
    uint32_t w[4];
    ptx::ldmatrix_x4(addr, w[0], w[1], w[2], w[3]);
#pragma unroll
    for (int P = 0; P < 2; ++P) {
      uint32_t ca[8], cb[8];
      split_int2(w[2 * P], ca);      // token g
      split_int2(w[2 * P + 1], cb);  // token g + 8
#pragma unroll
      for (int k = 0; k < 4; ++k)
        ptx::mma_16816(acc[P], ca[2 * k], cb[2 * k], ca[2 * k + 1], cb[2 * k + 1], bq[P][k][0],
                       bq[P][k][1]);
    }
  }
}

// PV of one 16-token sub-tile: O^T += c^T (p * scale)^T, and the min/l MMA.
// pb0/pb1 are the sub-tile's p as B fragments (tokens 2t, 2t+1 and 2t+8,
// 2t+9 of query g / 2), rounded to fp16, and pl0/pl1 the rest of p (p - pb,
// rounded to fp16): p is used as the sum of the two, so the weights carry
// about 22 bits.  p * scale goes in as the same two parts: the fp16 product,
// and what its rounding dropped plus p_lo * scale.
//   INT4 (and INT3 widened to INT4): each code MMA takes the rows of one group
//   and spends its 8 columns on 4 queries x the 2 parts: column n = 2 * query
//   + part, part 0 holding minus the fp16 product and part 1 the rest, so a
//   thread's accumulator pair (columns 2t, 2t+1) gives query t as [1] - [0].
//   oc[c][2G + jp]: group 2c + G; row g = dim 4g + 2jp (weight 1), row g+8 =
//   dim 4g + 2jp + 1 (weight 16).  The min/l MMA uses the same columns.
//   INT2: a group spans only 4 of the 8 lanes' code units, so its MMAs serve
//   two groups through the columns (n & 1 = group bit) and take each part
//   in a separate MMA; oc[c][pp]: rows g / g+8 = dims 64c + 8g + 2pp / +1,
//   group 2c + g/4 (fragments 0, 2 for g < 4; 1, 3 for g >= 4).
template <int BITS>
__device__ __forceinline__ void pv_subtile(uint32_t vc, const uint32_t* vp, int r0, int lane,
                                           uint32_t pb0, uint32_t pb1, uint32_t pl0, uint32_t pl1,
                                           float (&oc)[2][4][4], float (&mnacc)[4]) {
  const int g = lane >> 2, t = lane & 3;
  const int mj = lane >> 3, mi = lane & 7;
  const int lrow = r0 + (mj & 1) * 8 + mi;
  const int ra = r0 + 2 * t, rb = r0 + 2 * t + 8;  // this thread's B rows: ra, ra+1, rb, rb+1
  // A rows 0-3 = min of group g, row 8 = ones, others zero
  const int xg = g & 3;
  const uint32_t am0 = g < 4 ? ptx::prmt(vp[ra * NG + xg], vp[(ra + 1) * NG + xg], 0x7632u) : 0u;
  const uint32_t am2 = g < 4 ? ptx::prmt(vp[rb * NG + xg], vp[(rb + 1) * NG + xg], 0x7632u) : 0u;
  const uint32_t ones = g == 0 ? 0x3C003C00u : 0u;
  if constexpr (BITS == 4) {
    const bool rest = (g & 1) != 0;  // this thread's column holds the rest
    constexpr uint32_t kNeg = 0x80008000u;
    ptx::mma_16816(mnacc, am0, ones, am2, ones, rest ? pl0 : pb0 ^ kNeg, rest ? pl1 : pb1 ^ kNeg);
    // with these, the same three instructions give -fl16(pb * s) in part-0
    // columns and fl16(pl * s + (pb * s - fl16(pb * s))) in part-1 columns
    const uint32_t pbz0 = rest ? pb0 : 0u, pbz1 = rest ? pb1 : 0u;
    const uint32_t plz0 = rest ? pl0 : 0u, plz1 = rest ? pl1 : 0u;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      // w[0]/w[1]: group 2c, tokens (2t, 2t+1) / (2t+8, 2t+9), dims 4g..4g+3;
      // w[2]/w[3]: the same for group 2c+1
      const int chunk = 2 * c + (mj >> 1);
      const uint32_t addr = vc + lrow * 64 + ((chunk ^ ((lrow >> 1) & 3)) << 4);
      uint32_t w[4];
      ptx::ldmatrix_x4_trans(addr, w[0], w[1], w[2], w[3]);
      // scale/min of groups 2c, 2c+1 for the thread's four tokens
      const uint2 pa = *reinterpret_cast<const uint2*>(vp + ra * NG + 2 * c);
      const uint2 pa1 = *reinterpret_cast<const uint2*>(vp + (ra + 1) * NG + 2 * c);
      const uint2 pr = *reinterpret_cast<const uint2*>(vp + rb * NG + 2 * c);
      const uint2 pr1 = *reinterpret_cast<const uint2*>(vp + (rb + 1) * NG + 2 * c);
#pragma unroll
      for (int G = 0; G < 2; ++G) {
        const uint32_t sc0 = ptx::prmt(G ? pa.y : pa.x, G ? pa1.y : pa1.x, 0x5410u);
        const uint32_t sc1 = ptx::prmt(G ? pr.y : pr.x, G ? pr1.y : pr1.x, 0x5410u);
        const uint32_t u0 = ptx::hmul2_rn_u32(pb0, sc0);
        const uint32_t u1 = ptx::hmul2_rn_u32(pb1, sc1);
        const uint32_t b0 = ptx::hfma2_u32(plz0, sc0, ptx::hfma2_sub_u32(pbz0, sc0, u0));
        const uint32_t b1 = ptx::hfma2_u32(plz1, sc1, ptx::hfma2_sub_u32(pbz1, sc1, u1));
        uint32_t sa[4], sb[4];
        split_int4(w[2 * G], sa);      // tokens 2t, 2t+1
        split_int4(w[2 * G + 1], sb);  // tokens 2t+8, 2t+9
#pragma unroll
        for (int jp = 0; jp < 2; ++jp)
          ptx::mma_16816(oc[c][2 * G + jp], sa[2 * jp], sa[2 * jp + 1], sb[2 * jp], sb[2 * jp + 1],
                         b0, b1);
      }
    }
  } else {
    ptx::mma_16816(mnacc, am0, ones, am2, ones, pb0, pb1);
    ptx::mma_16816(mnacc, am0, ones, am2, ones, pl0, pl1);
    const int gb = g & 1;
    // w2[2c]/w2[2c+1] = tokens (2t, 2t+1) / (2t+8, 2t+9), dims 64c + 8g .. +7
    uint32_t w2[4];
    {
      const int chunk = mj >> 1;
      const uint32_t addr = vc + lrow * 32 + ((chunk ^ ((lrow >> 2) & 1)) << 4);
      ptx::ldmatrix_x4_trans(addr, w2[0], w2[1], w2[2], w2[3]);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      // p * scale of group 2c + (n & 1) for this thread's column n = g: the
      // rounded product of the fp16 parts, then (exact fma) what that rounding
      // dropped, plus p_lo * scale
      const int x = 2 * c + gb;
      const uint32_t sc0 = ptx::prmt(vp[ra * NG + x], vp[(ra + 1) * NG + x], 0x5410u);
      const uint32_t sc1 = ptx::prmt(vp[rb * NG + x], vp[(rb + 1) * NG + x], 0x5410u);
      const uint32_t bs0 = ptx::hmul2_rn_u32(pb0, sc0);
      const uint32_t bs1 = ptx::hmul2_rn_u32(pb1, sc1);
      const uint32_t bl0 = ptx::hfma2_u32(pl0, sc0, ptx::hfma2_sub_u32(pb0, sc0, bs0));
      const uint32_t bl1 = ptx::hfma2_u32(pl1, sc1, ptx::hfma2_sub_u32(pb1, sc1, bs1));
      uint32_t lo[8], hi[8];
      split_int2(w2[2 * c], lo);
      split_int2(w2[2 * c + 1], hi);
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
        ptx::mma_16816(oc[c][pp], lo[2 * pp], lo[2 * pp + 1], hi[2 * pp], hi[2 * pp + 1], bs0, bs1);
#pragma unroll
      for (int pp = 0; pp < 4; ++pp)
        ptx::mma_16816(oc[c][pp], lo[2 * pp], lo[2 * pp + 1], hi[2 * pp], hi[2 * pp + 1], bl0, bl1);
    }
  }
}

// ---------------------------------------------------------- residual ----

// fp16 split: rows [c0, c0 + kResRows) of the fp16 rows of one (sequence, KV
// head) (F16Rows), on the tensor cores.  Only the rows that take part are
// copied (zero-filled otherwise),
// so no stale bytes of unused slots enter the arithmetic.  Rows are padded to
// 272 bytes, which makes every ldmatrix conflict-free.  Warp w takes rows
// 16w .. 16w+15 as one sub-tile: S^T = K q^T (query columns duplicated, so each
// thread holds one query), softmax, O^T = V^T p^T, and writes its (m, l, o) to
// the merge scratch.
constexpr int kResRows = 64;
constexpr int kResStride = D * 2 + 16;  // bytes per row in shared memory

// The fp16 rows of one (sequence, KV head) as one index space: row j < Nr is
// slot j of the window ring, which takes part when its age (slot - ring head,
// mod Nr) lies in [age0, age1); row j >= Nr is sink row j - Nr, which takes part
// below sink_len.  Attention does not depend on the order of its tokens.
struct F16Rows {
  const __half* k_ring;  // this head's Nr window rows
  const __half* v_ring;
  const __half* k_sink;  // this head's Ns sink rows
  const __half* v_sink;
  int Nr, rh, age0, age1, ls;

  __device__ __forceinline__ bool valid(int j) const {
    if (j < Nr) {
      int age = j - rh;
      if (age < 0) age += Nr;
      return age >= age0 && age < age1;
    }
    return j - Nr < ls;
  }
  // row j of K (arr 0) or V (arr 1); an invalid j gives an in-bounds row that
  // is never read (its copy is zero-filled)
  __device__ __forceinline__ const __half* row(int arr, int j) const {
    const __half* ring = arr ? v_ring : k_ring;
    const __half* sink = arr ? v_sink : k_sink;
    if (!valid(j)) return Nr > 0 ? ring : sink;
    return j < Nr ? ring + (int64_t)j * D : sink + (int64_t)(j - Nr) * D;
  }
};

// Start the copies of the valid rows: K to rows 0..63, V to rows 64..127.
__device__ __forceinline__ void residual_issue(const F16Rows& fr, int c0, uint8_t* tiles) {
  const uint32_t tbase = ptx::smem_u32(tiles);
  for (int idx = threadIdx.x; idx < 2 * kResRows * (D / 8); idx += NTHREADS) {
    const int arr = idx / (kResRows * (D / 8));
    const int rem = idx % (kResRows * (D / 8));
    const int row = rem / (D / 8), chunk = rem % (D / 8);
    const int j = c0 + row;
    const __half* src = fr.row(arr, j) + chunk * 8;
    const bool ok = fr.valid(j);
    ptx::cp_async_16(tbase + (arr * kResRows + row) * kResStride + chunk * 16, src, ok ? 16u : 0u);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait for the copies, then attend (every thread of the CTA calls it).
__device__ __forceinline__ void residual_tc(const F16Rows& fr, int c0, uint8_t* tiles, int warp,
                                            int lane, const float (&q_s)[QB][D], float kq,
                                            MergeSmem& ms, bool merge) {
  const int g = lane >> 2, t = lane & 3;
  auto valid_slot = [&](int j) { return fr.valid(j); };
  const uint32_t tbase = ptx::smem_u32(tiles);
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  const int r0 = 16 * warp;
  const int mj = lane >> 3, mi = lane & 7;
  // ---- S^T = K q^T, one MMA per 16 head_dim values
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int row = r0 + (mj & 1) * 8 + mi;
    const uint32_t addr = tbase + row * kResStride + (16 * ks + (mj >> 1) * 8) * 2;
    uint32_t a0, a1, a2, a3;
    ptx::ldmatrix_x4(addr, a0, a1, a2, a3);
    const int qi = g >> 1, d0 = 16 * ks + 2 * t;
    const uint32_t b0 = ptx::pack_h2(q_s[qi][d0], q_s[qi][d0 + 1]);
    const uint32_t b1 = ptx::pack_h2(q_s[qi][d0 + 8], q_s[qi][d0 + 9]);
    ptx::mma_16816(acc, a0, a1, a2, a3, b0, b1);
  }
  // ---- softmax of query t over the warp's 16 rows
  const float s0 = valid_slot(c0 + r0 + g) ? acc[0] * kq : -INFINITY;
  const float s1 = valid_slot(c0 + r0 + g + 8) ? acc[2] * kq : -INFINITY;
  float m = fmaxf(s0, s1);
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
  const float mu = m == -INFINITY ? 0.f : m;
  // p in two fp16 parts (rounded, and the rest), used as their sum
  const float p0 = exp2f(s0 - mu), p1 = exp2f(s1 - mu);
  const uint32_t pk = ptx::pack_h2(p0, p1);
  const uint32_t pkl = ptx::pack_h2(p0 - half_lo(pk), p1 - half_hi(pk));
  const int srcA = (2 * t) * 4 + (g >> 1), srcB = (2 * t + 1) * 4 + (g >> 1);
  const uint32_t x0 = __shfl_sync(0xffffffffu, pk, srcA);
  const uint32_t x1 = __shfl_sync(0xffffffffu, pk, srcB);
  const uint32_t y0 = __shfl_sync(0xffffffffu, pkl, srcA);
  const uint32_t y1 = __shfl_sync(0xffffffffu, pkl, srcB);
  const uint32_t pb0 = ptx::prmt(x0, x1, 0x5410u);  // tokens 2t, 2t+1 of query g / 2
  const uint32_t pb1 = ptx::prmt(x0, x1, 0x7632u);  // tokens 2t+8, 2t+9
  const uint32_t pl0 = ptx::prmt(y0, y1, 0x5410u);
  const uint32_t pl1 = ptx::prmt(y0, y1, 0x7632u);
  // with merge, the warp's state already in ms (o, m, l of query t) is combined
  // with these rows': both are scaled to the larger max
  float al_old = 0.f, al_new = 1.f;
  if (merge) {
    const float m_old = ms.m[warp][t];
    const float mm = fmaxf(m_old, m);
    al_old = m_old == -INFINITY ? 0.f : exp2f(m_old - mm);
    al_new = m == -INFINITY ? 0.f : exp2f(mu - mm);
    if (mm == -INFINITY) al_new = 0.f;
  }
  // ---- O^T = V^T p^T, two MMAs (the parts of p) per 16 head_dim values; l =
  // sum of the same p
  float lacc[4] = {0.f, 0.f, 0.f, 0.f};
  constexpr uint32_t kOnes = 0x3C003C00u;
  ptx::mma_16816(lacc, kOnes, kOnes, kOnes, kOnes, pb0, pb1);
  ptx::mma_16816(lacc, kOnes, kOnes, kOnes, kOnes, pl0, pl1);
  const uint32_t vbase = tbase + kResRows * kResStride;
#pragma unroll
  for (int mb = 0; mb < D / 16; ++mb) {
    // matrices: tokens 0-7 | dims +0, tokens 0-7 | dims +8, tokens 8-15 | +0, 8-15 | +8
    const int row = r0 + (mj >> 1) * 8 + mi;
    const uint32_t addr = vbase + row * kResStride + (16 * mb + (mj & 1) * 8) * 2;
    uint32_t v0, v1, v2, v3;
    ptx::ldmatrix_x4_trans(addr, v0, v1, v2, v3);
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    ptx::mma_16816(o, v0, v1, v2, v3, pb0, pb1);
    ptx::mma_16816(o, v0, v1, v2, v3, pl0, pl1);
    float* dst = &ms.o[warp][t][16 * mb + g];
    dst[0] = merge ? fmaf(dst[0], al_old, o[0] * al_new) : o[0];
    dst[8] = merge ? fmaf(dst[8], al_old, o[2] * al_new) : o[2];
  }
  __syncwarp();  // every lane has read the old (m, l) of its query
  if (g == 0) {
    if (merge) {
      const float m_old = ms.m[warp][t];
      ms.l[warp][t] = fmaf(ms.l[warp][t], al_old, lacc[0] * al_new);
      ms.m[warp][t] = fmaxf(m_old, m);
    } else {
      ms.m[warp][t] = m;
      ms.l[warp][t] = lacc[0];
    }
  }
}

// --------------------------------------------------------------- kernel ----

// Grid (S, Hkv, B): split s < Sp streams packed tokens of (sequence b, KV head h)
// on the tensor cores; splits s >= Sp take 64 fp16 rows each (window ring slots,
// then sink rows).  Every split writes a partial (o, m, l); the last one of the
// head merges them.
//
// STEP: the same launch first appends one token per (sequence, KV head), as
// kvq_append does, and attends over the cache as it is after the append.  The
// packed splits only read rows that existed before the step.  The last residual
// split of each head does the append's writes: it quantizes the token that
// leaves the window (or, with no window, the new token) into packed slot
// packed_len with the pack kernel's quantizer, stores the new token in its ring
// slot, and attends over the window without the leaving token plus the new token
// (fp16) and the quantized one (dequantized in fp32).  The last head of a
// sequence to finish commits the counters.
template <int BITS, bool STEP, int CPS, int TT>
__global__ void __launch_bounds__(NTHREADS, CPS)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
                     const DecodeArgs a) {
  using G = Geo<BITS, CPS, TT>;
  constexpr int NSTAGE = G::NSTAGE;
  constexpr int T = G::T, NSUB = G::NSUB, WR = G::WR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full_bar[NSTAGE];
  __shared__ int s_rel[NSTAGE];        // warps done with the stage's current tile
  __shared__ int s_last_tile[NSTAGE];  // last tile issued into each stage (-1: none)
  __shared__ float q_s[QB][D];
  __shared__ float qsum_s[QB][NG];  // sum of q over each group
  // range lo, hi, ring head, step flags, packed_len, res_len, sink_len, and the
  // fp16 rows' age range of a packed split that also takes them
  __shared__ int s_rng[9];
  __shared__ volatile int s_abort;
  __shared__ int s_last;
  __shared__ uint32_t s_ref[QB];  // the head's reference max per query (float bits + 1; 0: unknown)
  __shared__ int s_pages[kPagePrefetch];  // paged caches: the split's first page ids
  __shared__ uint32_t s_bad[NSTAGE];      // paged caches: bit p = page p of the stage's tile is bad

  const int s = blockIdx.x;
  const int h = blockIdx.y;  // one query block per KV head (gq <= 4)
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;  // MMA group id
  const int t = lane & 3;   // thread in group
  const bool res_cta = s >= a.Sp;  // an fp16 split: window and sink rows
  // in a grid of several waves the last packed split of the (sequence, KV head)
  // also takes its fp16 rows (and, in a fused step, the append)
  const bool fold_cta = a.fold != 0 && s == a.Sp - 1;
  const int64_t bh = (int64_t)b * a.Hkv + h;
  const int f0 = kResRows * (s - a.Sp);  // an fp16 split's first row
  const bool has_f16 = a.Nr + a.Ns > 0;
  const uint64_t wait_ns = (uint64_t)a.wait_limit_us * 1000u;
  // testing hook (off unless the host armed it): the first tile of split 0 of
  // (sequence 0, KV head 0) expects more bytes than its copies deliver
  const uint32_t fault_tx = (s == 0 && h == 0 && b == 0) ? a.fault_tx : 0u;
  // the fp16 rows of this (sequence, KV head), ranges from the counters
  auto f16_rows = [&]() {
    const int ia = res_cta ? 0 : 7;  // where plan() left the window's age range
    F16Rows fr;
    fr.k_ring = a.k_res + bh * a.Nr * D;
    fr.v_ring = a.v_res + bh * a.Nr * D;
    fr.k_sink = a.k_sink + bh * a.Ns * D;
    fr.v_sink = a.v_sink + bh * a.Ns * D;
    fr.Nr = a.Nr;
    fr.rh = s_rng[2];
    fr.age0 = s_rng[ia];
    fr.age1 = s_rng[ia + 1];
    fr.ls = s_rng[6];
    return fr;
  };

  // Prologue that touches no global memory; the rest waits for the grid this
  // launch depends on (the append of the same step) to complete.
  if (threadIdx.x == 0) {
    for (int st = 0; st < NSTAGE; ++st) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[st]), 1);
      s_rel[st] = 0;
      s_last_tile[st] = -1;
    }
    s_abort = 0;
    for (int i = 0; i < QB; ++i) s_ref[i] = 0u;
    ptx::fence_mbar_init();
    if (!res_cta) {
      ptx::prefetch_tensormap(&tm_kc);
      ptx::prefetch_tensormap(&tm_vc);
    }
  }
  // A launch that depends on this one programmatically (the next step) may
  // start filling the SMs this grid frees; it waits for this grid before it
  // touches anything this grid writes.
  asm volatile("griddepcontrol.launch_dependents;");

  int i0 = 0, i1 = 0, ntiles = 0, row0 = 0;
  uint32_t err_bits = 0;
  // packed rows in the codes / params arrays (bulk copies must stay inside)
  const int64_t prows = a.rm.paged ? (int64_t)a.rm.npages * a.Hkv * kPage
                                   : (int64_t)gridDim.z * a.Hkv * a.cap;
  constexpr uint32_t kParRow = NG * 4;  // param bytes per packed row
  auto issue = [&](int tile) {
    const int st = tile % NSTAGE;
    s_last_tile[st] = tile;
    uint8_t* base = smem + (size_t)st * G::STAGE;
    const uint32_t fb = ptx::smem_u32(&full_bar[st]);
    if (!a.rm.paged) {
      // y lies inside this head's rows; the params copy stops at the array end
      // (rows past the split end are masked)
      const int y = row0 + tile * T;
      const uint32_t pbytes = (uint32_t)min((int64_t)T, prows - y) * kParRow;
      ptx::mbar_arrive_expect_tx(fb, 2 * G::CODE_TILE + 2 * pbytes + (tile == 0 ? fault_tx : 0u));
      ptx::tma_load_2d(ptx::smem_u32(base + G::KC), &tm_kc, 0, y, fb);
      ptx::tma_load_2d(ptx::smem_u32(base + G::VC), &tm_vc, 0, y, fb);
      ptx::bulk_load(ptx::smem_u32(base + G::KP), a.k_params + (int64_t)y * NG, pbytes, fb);
      ptx::bulk_load(ptx::smem_u32(base + G::VP), a.v_params + (int64_t)y * NG, pbytes, fb);
    } else {
      // the tile's pages (i0 is a page boundary), 32 rows of each array apiece;
      // stage rows past the split's last page keep stale bytes, masked like
      // any rows past the split end
      constexpr int kPerTile = T / kPage;
      const int j0 = tile * kPerTile;
      const int np = min(kPerTile, (i1 - i0 + kPage - 1) / kPage - j0);
      int ys[kPerTile];
      uint32_t bytes = tile == 0 ? fault_tx : 0u, bad = 0;
      for (int p = 0; p < np; ++p) {
        const int j = j0 + p;
        const int pg = j < kPagePrefetch ? s_pages[j] : a.rm.page_of(b, i0 / kPage + j);
        // a page outside the pool: its codes read zeros (TMA fill), no params
        // are copied, and the page is flagged
        ys[p] = (pg >= 0 && pg < a.rm.npages) ? (pg * a.Hkv + h) * kPage : -kPage;
        bytes += 2 * kPage * G::RB + (ys[p] >= 0 ? 2 * kPage * kParRow : 0);
        if (ys[p] < 0) {
          set_error(a.err_word, KVQ_ERRBIT_BADPAGE);
          bad |= 1u << p;
        }
      }
      // the consumers skip a bad page's rows (read after the barrier completes)
      s_bad[st] = bad;
      ptx::mbar_arrive_expect_tx(fb, bytes);
      for (int p = 0; p < np; ++p) {
        const int y = ys[p];
        ptx::tma_load_2d(ptx::smem_u32(base + G::KC + p * kPage * G::RB), &tm_kc, 0, y, fb);
        ptx::tma_load_2d(ptx::smem_u32(base + G::VC + p * kPage * G::RB), &tm_vc, 0, y, fb);
        if (y >= 0) {
          ptx::bulk_load(ptx::smem_u32(base + G::KP + p * kPage * kParRow),
                         a.k_params + (int64_t)y * NG, kPage * kParRow, fb);
          ptx::bulk_load(ptx::smem_u32(base + G::VP + p * kPage * kParRow),
                         a.v_params + (int64_t)y * NG, kPage * kParRow, fb);
        }
      }
    }
  };
  // Thread 0: read the counters, cut this split's range and (tma_first) start
  // its first NSTAGE tiles with TMA copies.
  auto plan = [&](bool tma_first) {
    const int Lp = a.packed_len[b];
    const int Lr = a.res_len[b];
    // fused step: the append packs a token when the window is full (or absent),
    // and changes nothing when that would overflow the packed capacity
    const bool pack_now = a.Nr == 0 || Lr == a.Nr;
    const bool full = STEP && pack_now && Lp >= a.cap;
    const bool adds = STEP && !full;
    const int Ls = a.Ns > 0 ? a.sink_len[b] : 0;
    int r0_, r1_, xflags = 0;
    if (!res_cta) {
      r0_ = (int)((int64_t)Lp * s / a.Sp);
      r1_ = (int)((int64_t)Lp * (s + 1) / a.Sp);
      if (a.rm.paged) {  // splits start on page boundaries
        r0_ = r0_ / kPage * kPage;
        r1_ = s + 1 == a.Sp ? Lp : r1_ / kPage * kPage;
      }
    }
    // window tokens of age [jlo, Lr) take part (a flushed oldest token leaves
    // the window); residual split sr holds ring slots [64 sr, 64 sr + 64)
    const int jlo = (adds && a.Nr > 0 && pack_now) ? 1 : 0;
    if (res_cta) {
      const int Sr = a.S - a.Sp, sr = s - a.Sp;
      r0_ = jlo;
      r1_ = Lr;
      // bit 0: the new token joins the window; bit 1: a token is packed into slot Lp
      if (adds && sr == Sr - 1) xflags = (a.Nr > 0 ? 1 : 0) | (pack_now ? 2 : 0);
    }
    if (fold_cta && adds) xflags = (a.Nr > 0 ? 1 : 0) | (pack_now ? 2 : 0);
    s_rng[7] = jlo;
    s_rng[8] = Lr;
    s_rng[0] = r0_;
    s_rng[1] = r1_;
    s_rng[2] = a.res_head[b];  // every split: the last one to finish commits the step
    s_rng[3] = xflags;
    s_rng[4] = Lp;
    s_rng[5] = Lr;
    s_rng[6] = Ls;
    if (s == 0 && Lp + Lr + Ls == 0 && !adds) err_bits |= KVQ_ERRBIT_EMPTY;
    if (full && s == 0 && h == 0) err_bits |= KVQ_ERRBIT_CAPACITY;
    if (!res_cta) {
      i0 = r0_;
      i1 = r1_;
      ntiles = (i1 - i0 + T - 1) / T;
      row0 = (int)(bh * a.cap + i0);  // first packed row of this split (TMA y, contiguous)
      if (a.rm.paged) {
        const int npg = min((i1 - i0 + kPage - 1) / kPage, kPagePrefetch);
        for (int j = 0; j < npg; ++j) s_pages[j] = a.rm.page_of(b, i0 / kPage + j);
      }
      if (tma_first)
        for (int tile = 0; tile < ntiles && tile < NSTAGE; ++tile) issue(tile);
    }
  };
  // With the caller's word that the kernel before this launch does not write
  // this cache (KVQ_STEP_EARLY_CACHE_READ), thread 0 reads the counters and cuts
  // the ranges before waiting for that kernel, so the copies can start the
  // moment the wait returns.  The copies themselves are issued after the wait:
  // copies a dependent launch issues before it (bulk, tensor, cp.async, even
  // plain loads of data that must come from memory) were measured to be served
  // only once the launch it depends on had completed, and queued ahead of that
  // launch's last memory operations they delayed its completion and with it
  // the wait.  An L2 prefetch of each split's tile 0 alone (9 of the 42 MB a
  // 32K INT4 step reads) is cheap enough there: in a grid of one wave it lets
  // tile 0 land sooner.  q and the new token are read after the wait.
  const bool early = STEP && a.early != 0;
  if (early && threadIdx.x == 0) {
    plan(false);
    if (!res_cta && !a.rm.paged && !a.fold && ntiles > 0) {
      const uint32_t rows = (uint32_t)min(T, i1 - i0);  // this head's rows from row0
      ptx::prefetch_l2(a.k_codes + (int64_t)row0 * G::RB, rows * G::RB);
      ptx::prefetch_l2(a.v_codes + (int64_t)row0 * G::RB, rows * G::RB);
      ptx::prefetch_l2(a.k_params + (int64_t)row0 * NG, rows * kParRow);
      ptx::prefetch_l2(a.v_params + (int64_t)row0 * NG, rows * kParRow);
    }
  }
  grid_dependency_wait();

  // The small loads go first -- q by every thread, the lengths by thread 0 --
  // so they are not queued behind the bulk tile copies.  QB * D / 128 = 4 halves
  // per thread; query heads past gq (gq < 4) stay zero.
  const int q_i = (threadIdx.x * 4) / D;
  uint2 qraw = make_uint2(0, 0);
  if (q_i < a.gq)
    qraw = *reinterpret_cast<const uint2*>(a.q + ((int64_t)b * a.Hq + h * a.gq) * D + threadIdx.x * 4);
  if (threadIdx.x == 0) {
    if (!early) plan(true);
    else if (!res_cta)  // ranges read before the wait: start the first tiles now
      for (int tile = 0; tile < ntiles && tile < NSTAGE; ++tile) issue(tile);
    if (err_bits) set_error(a.err_word, err_bits);
  }
  {
    const int e = (threadIdx.x * 4) % D;
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&qraw.x));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&qraw.y));
    q_s[q_i][e] = f01.x;
    q_s[q_i][e + 1] = f01.y;
    q_s[q_i][e + 2] = f23.x;
    q_s[q_i][e + 3] = f23.y;
  }
  __syncthreads();  // barriers initialised, range and q staged
  const float kq = a.qk_scale_log2;
  MergeSmem& ms = *reinterpret_cast<MergeSmem*>(smem);

  if (res_cta && has_f16) residual_issue(f16_rows(), f0, smem + kResTilesOff);

  // extra tokens of a fused step, fp32: [K, V][new token, packed token][D]
  float* xbuf = reinterpret_cast<float*>(smem + sizeof(MergeSmem));
  auto append_work = [&]() {
    // the append's writes for this (sequence, KV head): warp 0 the K row, warp
    // 1 the V row, lane l < 16 holding values 8l .. 8l+7 (as in kvq_append)
    const int which = warp;
    const int xflags = s_rng[3], rh = s_rng[2], Lp = s_rng[4], Lr = s_rng[5];
    const bool active = lane < D / 8;
    uint4 nv = make_uint4(0, 0, 0, 0);
    if (active)
      nv = __ldg(reinterpret_cast<const uint4*>((which ? a.v_new : a.k_new) + bh * D) + lane);
    float* xb = xbuf + which * 2 * D;
    if (xflags & 2) {
      // the oldest window token (or, with no window, the new one) -> slot Lp
      uint4 src = nv;
      if (a.Nr > 0 && active)
        src = *reinterpret_cast<const uint4*>(a.w_res[which] + (bh * a.Nr + rh) * D + lane * 8);
      uint32_t prm, asym = 1;
      const uint32_t packed = quantize_quad<BITS>(src, prm, a.hybrid != 0, &asym);
      const uint32_t modes = __ballot_sync(0xffffffffu, (lane & 3) == 0 && asym);
      const int64_t row = a.rm.row(b, h, Lp);  // warp-uniform
      if (row < 0 && lane == 0) {
        // a page outside the pool: nothing is stored and, as a decode after
        // kvq_append would, the token is not attended
        set_error(a.err_word, KVQ_ERRBIT_BADPAGE);
        s_rng[3] = xflags & ~2;
      }
      if (a.hybrid && lane == 0 && row >= 0) a.w_modes[which][row] = mode_byte(modes, 0, NG);
      {
        const int gi = lane >> 2, quad = lane & 3;
        store_group_codes<BITS>(a.w_codes[which] + (row < 0 ? 0 : row) * a.row_bytes + gi * (4 * BITS),
                                packed, quad, active && row >= 0);
        if (active && row >= 0 && quad == 0) a.w_params[which][row * NG + gi] = prm;
      }
      if (active) {  // the packed token as it is attended, dequantized in fp32
        const float sc = half_lo(prm), mn = half_hi(prm);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          xb[D + lane * 8 + j] = fmaf((float)((packed >> (BITS * j)) & ((1u << BITS) - 1u)), sc, mn);
      }
    }
    if ((xflags & 1) && active) {
      // the new token takes the leaving token's slot, or the next free one
      float x[8];
      unpack8_f16(nv, x);
#pragma unroll
      for (int j = 0; j < 8; ++j) xb[lane * 8 + j] = x[j];
      const int slot = (xflags & 2) ? rh : (rh + Lr) % a.Nr;
      *reinterpret_cast<uint4*>(a.w_res[which] + (bh * a.Nr + slot) * D + lane * 8) = nv;
    }
  };
  auto join_extra = [&]() {
      // the appended tokens (new fp16 token, quantized token), staged in xbuf by
      // warps 0 and 1 before the barrier above, join warp 0's state; lane = four
      // head_dim values
      const int xflags = s_rng[3];
      __syncwarp();
      if (xflags != 0 && warp == 0) {
#pragma unroll
        for (int i = 0; i < QB; ++i) {
          float rm = ms.m[0][i], rl = ms.l[0][i];
          float ro[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) ro[jj] = ms.o[0][i][lane * 4 + jj];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (!(xflags & (1 << e))) continue;
            float part = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) part = fmaf(xbuf[e * D + lane * 4 + jj], q_s[i][lane * 4 + jj], part);
            const float v = warp_sum(part) * kq;
            const float mnew = fmaxf(rm, v);
            const float al = exp2f(rm - mnew);
            const float pe = exp2f(v - mnew);
            rl = fmaf(rl, al, pe);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) ro[jj] = fmaf(pe, xbuf[2 * D + e * D + lane * 4 + jj], ro[jj] * al);
            rm = mnew;
          }
          __syncwarp();
          if (lane == 0) {
            ms.m[0][i] = rm;
            ms.l[0][i] = rl;
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) ms.o[0][i][lane * 4 + jj] = ro[jj];
        }
      }
  };
  if (STEP && res_cta && warp < 2 && s_rng[3] != 0) append_work();

  if (res_cta) {
    // ------------------------------------------------ fp16-token split
    uint8_t* tiles = smem + kResTilesOff;
    if (has_f16) {
      residual_tc(f16_rows(), f0, tiles, warp, lane, q_s, kq, ms, false);
    } else {  // no fp16 rows (the split only takes a fused step's packed token)
      __syncthreads();  // warp 1's V row of the extra token is staged
      if (lane < QB) {
        ms.m[warp][lane] = -INFINITY;
        ms.l[warp][lane] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < QB; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) ms.o[warp][i][lane * 4 + jj] = 0.f;
    }
    if (STEP) join_extra();
  } else {
    // ---------------------------------------------------- packed-token split
    {
      // sum of q per (query, group), eight threads each
      const int sidx = threadIdx.x >> 3, part = threadIdx.x & 7;
      const int qi = sidx >> 2, grp = sidx & 3;
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) sum += q_s[qi][grp * kGroup + part * 4 + k];
#pragma unroll
      for (int o = 1; o <= 4; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (part == 0) qsum_s[qi][grp] = sum;
    }
    i0 = s_rng[0];
    i1 = s_rng[1];
    const int npk = i1 - i0;
    ntiles = (npk + T - 1) / T;
    row0 = (int)(bh * a.cap + i0);
    __syncthreads();  // qsum_s ready
    const float kq24 = kq * kTwo24;  // scores come out of the fix-up times 2^-24

    float m_ref = -INFINITY;  // running max of query t, log2 units
    float oc[2][4][4];        // O^T accumulators (layout at pv_subtile), times 2^-24
    float mnacc[4];           // C-fragment of the min/l MMA
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) oc[x][m][r] = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) mnacc[r] = 0.f;

    // q as B fragments of the K-side MMA.  Column n = 2 * query + group bit:
    // even columns take the pair's first group, odd ones its second, so the
    // accumulator a thread holds (columns 2t, 2t+1) is query t for both groups.
    // bq[P][s][0] covers k rows 2t, 2t+1 and bq[P][s][1] rows 2t+8, 2t+9, each
    // divided by the weight of the code position it meets.
    uint32_t bq[2][4][2];
    float qs_t[NG];  // query t: group sums of q, times 2^-24 like the accumulators
#pragma unroll
    for (int x = 0; x < NG; ++x) qs_t[x] = qsum_s[t][x] * (1.f / kTwo24);
    {
      const int qi = g >> 1;
#pragma unroll
      for (int P = 0; P < 2; ++P) {
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          if (G::CB == 4) {
            // k rows 2t, 2t+1 <- group P, d = 8t + st (+4); 2t+8, 2t+9 <- group P+2
            const int da = 32 * P + 8 * t + st;
            const int db = 32 * (P + 2) + 8 * t + st;
            const float iw = 1.f / w4_weight(st);
            bq[P][st][0] = (g & 1) == 0 ? ptx::pack_h2(q_s[qi][da] * iw, q_s[qi][da + 4] * iw) : 0u;
            bq[P][st][1] = (g & 1) == 1 ? ptx::pack_h2(q_s[qi][db] * iw, q_s[qi][db + 4] * iw) : 0u;
          } else {
            // thread t's codes: d = 64P + 16t + j, group 2P + (t >> 1); k rows
            // 2t, 2t+1 <- j = 2st, 2st+8; 2t+8, 2t+9 <- j = 2st+1, 2st+9
            const bool nz = (g & 1) == (t >> 1);
            const int d0 = 64 * P + 16 * t + 2 * st;
            const float iw0 = 1.f / w2_weight(2 * st), iw1 = 1.f / w2_weight(2 * st + 1);
            bq[P][st][0] = nz ? ptx::pack_h2(q_s[qi][d0] * iw0, q_s[qi][d0 + 8] * iw0) : 0u;
            bq[P][st][1] = nz ? ptx::pack_h2(q_s[qi][d0 + 1] * iw1, q_s[qi][d0 + 9] * iw1) : 0u;
          }
        }
      }
    }

    // After its first tile, warp 0 offers its running max of each query as the
    // head's reference (first offer wins); the answer is only needed at the end.
    uint32_t ref_cas = 0u;
    float ref_mine = 0.f;
    bool ref_offered = false;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int st = tile % NSTAGE;
      if (!ptx::mbar_wait_bounded(ptx::smem_u32(&full_bar[st]), (tile / NSTAGE) & 1, wait_ns)) {
        if (lane == 0) set_error(a.err_word, KVQ_ERRBIT_TIMEOUT);
        s_abort = 1;
        break;
      }
      uint8_t* base = smem + (size_t)st * G::STAGE;
      const int wrow = WR * warp;                         // first row of this warp
      // rows of this warp still ours; in a paged cache (128-token tiles) a
      // warp's 32 rows are one page, and none of a page outside the pool takes part
      int nvalid = min(npk - tile * T - wrow, WR);
      if (a.rm.paged && ((s_bad[st] >> (wrow / kPage)) & 1u)) nvalid = 0;
      if (nvalid > 0) {
        // rows past the split end may hold anything: zero their params so no
        // Inf/NaN reaches the arithmetic (their scores are masked anyway)
        if (nvalid < WR) {
          for (int r = lane; r < WR; r += 32)
            if (r >= nvalid) {
              reinterpret_cast<uint4*>(base + G::KP)[wrow + r] = make_uint4(0, 0, 0, 0);
              reinterpret_cast<uint4*>(base + G::VP)[wrow + r] = make_uint4(0, 0, 0, 0);
            }
          __syncwarp();
        }
        uint32_t kc = ptx::smem_u32(base + G::KC);
        uint32_t vc = ptx::smem_u32(base + G::VC);
        const uint32_t* kp = reinterpret_cast<const uint32_t*>(base + G::KP);
        const uint32_t* vp = reinterpret_cast<const uint32_t*>(base + G::VP);
        int crow = wrow;  // this warp's first row in the code tiles it reads
        if constexpr (BITS == 3) {
          // widen the warp's rows of K and V codes (lane = row) into its own
          // INT4 buffers; the params stay in the stage (rows offset by wrow)
          uint8_t* xk = smem + (size_t)NSTAGE * G::STAGE + (size_t)warp * (2 * WR * 64);
          for (int r = lane; r < WR; r += 32) {
            widen_row3(base + G::KC + (wrow + r) * G::RB, ptx::smem_u32(xk), r);
            widen_row3(base + G::VC + (wrow + r) * G::RB, ptx::smem_u32(xk + WR * 64), r);
          }
          __syncwarp();
          kc = ptx::smem_u32(xk);
          vc = ptx::smem_u32(xk + WR * 64);
          vp += wrow * NG;
          crow = 0;
        }

        // ---------------- QK for both sub-tiles
        float acc[NSUB][2][4];
#pragma unroll
        for (int u = 0; u < NSUB; ++u) qk_subtile<G::CB>(kc, crow + 16 * u, lane, bq, acc[u]);

        // fix-up, fp32: acc_g = 2^-24 sum c q, so 2^-24 s = sum_g scale_g acc_g +
        // min_g (2^-24 qsum_g) for query t; rows past the split end masked
        float sv[NSUB][2];  // [sub-tile][row g / g+8]
#pragma unroll
        for (int u = 0; u < NSUB; ++u) {
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int row = wrow + 16 * u + g + 8 * rr;
            const uint4 pr = reinterpret_cast<const uint4*>(kp)[row];
            const uint32_t prm[NG] = {pr.x, pr.y, pr.z, pr.w};
            float acc_s = 0.f;
#pragma unroll
            for (int P = 0; P < 2; ++P) {
              const int ga = G::CB == 4 ? P : 2 * P;
              const int gb = G::CB == 4 ? P + 2 : 2 * P + 1;
              acc_s = fmaf(half_lo(prm[ga]), acc[u][P][2 * rr], acc_s);
              acc_s = fmaf(half_lo(prm[gb]), acc[u][P][2 * rr + 1], acc_s);
            }
#pragma unroll
            for (int x = 0; x < NG; ++x) acc_s = fmaf(half_hi(prm[x]), qs_t[x], acc_s);
            sv[u][rr] = (16 * u + g + 8 * rr < nvalid) ? acc_s : -INFINITY;
          }
        }

        // ---------------- online softmax over the warp's 32 rows (lazy rescale).
        // The running max of query t moves only when one of its rows lies more
        // than 8 above it; each thread checks its own rows, and only then does
        // the warp reduce the max over the lanes of each query.
        float mown = fmaxf(sv[0][0], sv[0][1]);
#pragma unroll
        for (int u = 1; u < NSUB; ++u) mown = fmaxf(mown, fmaxf(sv[u][0], sv[u][1]));
        mown *= kq24;
        if (__any_sync(0xffffffffu, mown > m_ref + 8.f)) {
          float mloc = mown;
          mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 4));
          mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 8));
          mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16));
          const bool need = mloc > m_ref + 8.f;  // the same for every lane of query t
          const float mnew = need ? mloc : m_ref;
          const float al = need ? exp2f(m_ref - mnew) : 1.f;
          m_ref = mnew;
          // every O accumulator of this thread is query t
#pragma unroll
          for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
              for (int r = 0; r < 4; ++r) oc[x][m][r] *= al;
#pragma unroll
          for (int r = 0; r < 4; ++r) mnacc[r] *= al;
        }
        if (tile == 0 && warp == 0 && lane < QB && a.S > 1) {
          ref_mine = m_ref;
          ref_cas = atomicCAS(&a.ref_max[bh * QB + lane], 0u, __float_as_uint(m_ref) + 1u);
          ref_offered = true;
        }
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        // p as the PV B fragments, in two fp16 parts (p rounded, and the rest):
        // thread (g, t) needs p(query g / 2, tokens 2t, 2t+1, 2t+8, 2t+9); lane
        // 4 * token + query holds that query for rows token and token + 8 of the
        // sub-tile
        const int srcA = (2 * t) * 4 + (g >> 1);
        const int srcB = (2 * t + 1) * 4 + (g >> 1);
#pragma unroll
        for (int u = 0; u < NSUB; ++u) {
          // (weights below 2^-126 of the running max's are flushed to zero)
          const float p0 = ptx::ex2_ftz(fmaf(sv[u][0], kq24, -mu));
          const float p1 = ptx::ex2_ftz(fmaf(sv[u][1], kq24, -mu));
          const uint32_t pk = ptx::pack_h2(p0, p1);
          const uint32_t pkl = ptx::pack_h2(p0 - half_lo(pk), p1 - half_hi(pk));  // exact differences
          const uint32_t x0 = __shfl_sync(0xffffffffu, pk, srcA);  // (p(2t), p(2t+8))
          const uint32_t x1 = __shfl_sync(0xffffffffu, pk, srcB);  // (p(2t+1), p(2t+9))
          const uint32_t y0 = __shfl_sync(0xffffffffu, pkl, srcA);
          const uint32_t y1 = __shfl_sync(0xffffffffu, pkl, srcB);
          const uint32_t pb0 = ptx::prmt(x0, x1, 0x5410u);  // tokens 2t, 2t+1
          const uint32_t pb1 = ptx::prmt(x0, x1, 0x7632u);  // tokens 2t+8, 2t+9
          const uint32_t pl0 = ptx::prmt(y0, y1, 0x5410u);
          const uint32_t pl1 = ptx::prmt(y0, y1, 0x7632u);
          pv_subtile<G::CB>(vc, vp, crow + 16 * u, lane, pb0, pb1, pl0, pl1, oc, mnacc);
        }
      }
      __syncwarp();
      // Release the stage.  The warp that releases it last refills it with tile
      // + NSTAGE straight away: nobody waits for the slowest warp.
      if (lane == 0) {
        // release: this warp's reads of the stage come first; acquire: the
        // warp that completes the count sees the others' releases
        if (ptx::atom_add_acq_rel_cta(ptx::smem_u32(&s_rel[st]), 1u) == NCW - 1) {
          s_rel[st] = 0;
          const int next = tile + NSTAGE;
          if (next < ntiles && !s_abort) {
            ptx::fence_proxy_async_shared();  // generic reads before the TMA overwrite
            issue(next);
          }
        }
      }
      __syncwarp();
      if (s_abort) break;
    }
    __syncthreads();  // the stage ring is idle from here on: reuse it for the merge
    // Copies still in flight (only after an abort: otherwise every issued tile
    // was consumed) land before the ring is reused.
    if (s_abort) {  // CTA-uniform after the barrier
      if (threadIdx.x == 0) {
        for (int st = 0; st < NSTAGE; ++st)
          if (s_last_tile[st] >= 0)
            ptx::mbar_wait_bounded(ptx::smem_u32(&full_bar[st]), (s_last_tile[st] / NSTAGE) & 1, wait_ns);
      }
      __syncthreads();
    }
    if (s_abort) {
      // a wait ran out: this split contributes nothing (it still takes its
      // ticket below, so the head's merge and the workspace stay consistent)
      m_ref = -INFINITY;
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) oc[x][m][r] = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) mnacc[r] = 0.f;
    }
    if (ref_offered) s_ref[lane] = ref_cas == 0u ? __float_as_uint(ref_mine) + 1u : ref_cas;
    // per group x and query t, sum p min_x to shared memory first; then the
    // outputs O = 2^24 oc / weight + sum p min (the layouts are at pv_subtile;
    // INT4 columns hold minus the first part and the rest)
    if (g < 4) ms.mn[warp][g][t] = G::CB == 4 ? mnacc[1] - mnacc[0] : mnacc[0];
    if (g == 0) {
      ms.l[warp][t] = G::CB == 4 ? mnacc[3] - mnacc[2] : mnacc[2];
      ms.m[warp][t] = m_ref;
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (G::CB == 4) {
          const int grp = 2 * c + (j >> 1), jp = j & 1;
          const float mnv = ms.mn[warp][grp][t];
          const int d0 = 32 * grp + 4 * g + 2 * jp;
          ms.o[warp][t][d0] = fmaf(oc[c][j][1] - oc[c][j][0], kTwo24 / w4_weight(2 * jp), mnv);
          ms.o[warp][t][d0 + 1] = fmaf(oc[c][j][3] - oc[c][j][2], kTwo24 / w4_weight(2 * jp + 1), mnv);
        } else {
          const int hb = g >> 2;
          const float mnv = ms.mn[warp][2 * c + hb][t];
          const int d0 = 64 * c + 8 * g + 2 * j;
          ms.o[warp][t][d0] = fmaf(hb ? oc[c][j][1] : oc[c][j][0], kTwo24 / w2_weight(2 * j), mnv);
          ms.o[warp][t][d0 + 1] = fmaf(hb ? oc[c][j][3] : oc[c][j][2], kTwo24 / w2_weight(2 * j + 1), mnv);
        }
      }
  }

  if (fold_cta) {
    // this split also takes the fp16 rows (window, then sink) and, in a fused
    // step, the append, as an fp16 split would; the stage ring is idle
    __syncthreads();  // every warp's packed state is in ms
    uint8_t* tiles = smem + kResTilesOff;
    if (has_f16) residual_issue(f16_rows(), 0, tiles);
    if (STEP && warp < 2 && s_rng[3] != 0) append_work();
    if (has_f16) {
      for (int c0 = 0; c0 < a.Nr + a.Ns; c0 += kResRows) {
        if (c0 > 0) {
          __syncthreads();  // the previous rows are read
          residual_issue(f16_rows(), c0, tiles);
        }
        residual_tc(f16_rows(), c0, tiles, warp, lane, q_s, kq, ms, true);
      }
    } else {
      __syncthreads();  // warp 1's V row of the extra token is staged
    }
    if (STEP) join_extra();
  }

  // ---------------- merge the four warps' states.  The split's partial (o, m, l)
  // goes to the workspace for the fallback merge, and the same state, scaled to
  // the head's reference max, is added into the head's fp32 accumulators.
  __syncthreads();
  const int64_t pidx = bh * a.S + s;
  {
    const int i = warp;              // query
    const int e = lane * 4;          // four head_dim values
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, ms.m[w][i]);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < NCW; ++w) {
        const float f = exp2f(ms.m[w][i] - M);
        if (f > 0.f) {
          const float4 ow = *reinterpret_cast<const float4*>(&ms.o[w][i][e]);
          o.x = fmaf(ow.x, f, o.x);
          o.y = fmaf(ow.y, f, o.y);
          o.z = fmaf(ow.z, f, o.z);
          o.w = fmaf(ow.w, f, o.w);
          lsum = fmaf(ms.l[w][i], f, lsum);
        }
      }
    }
    if (a.S == 1) {
      // the head's only split: its state is the result (no partials, no
      // accumulators, no ticket)
      if (i < a.gq) {
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        store_out4(a, ((int64_t)b * a.Hq + h * a.gq + i) * D + e,
                   make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv));
      }
    } else {
    *reinterpret_cast<float4*>(a.o_part + (pidx * QB + i) * D + e) = o;
    if (lane == 0) a.ml_part[pidx * QB + i] = make_float2(M, lsum);
    if (M > -INFINITY) {  // warp-uniform
      uint32_t ref = s_ref[i];
      if (ref == 0u) {  // this split offered nothing yet: offer (or learn) now
        uint32_t r = 0u;
        if (lane == 0) {
          const uint32_t mine = __float_as_uint(M) + 1u;
          const uint32_t old = atomicCAS(&a.ref_max[bh * QB + i], 0u, mine);
          r = old == 0u ? mine : old;
        }
        ref = __shfl_sync(0xffffffffu, r, 0);
      }
      const float dm = M - __uint_as_float(ref - 1u);
      if (dm > kRefSlack) {
        if (lane == 0) ptx::red_or_u32(&a.fb_flag[bh], 1u);  // too far above: exact merge instead
      } else {
        const float g = exp2f(dm);
        ptx::red_add_v4(a.o_acc + (bh * QB + i) * D + e, o.x * g, o.y * g, o.z * g, o.w * g);
        if (lane == 0) ptx::red_add_f32(&a.l_acc[bh * QB + i], lsum * g);
      }
    }
    }
  }
  // Fused step: once every split of a head has read the counters, the head takes
  // a ticket on its sequence; the last head of the sequence commits the append's
  // counters, computed from the values this CTA read at its start.
  auto commit_step = [&](unsigned seq_ticket) {
    if (STEP && threadIdx.x == 0 && seq_ticket == (unsigned)(a.Hkv - 1)) {
      const int Lp = s_rng[4], Lr = s_rng[5], rh = s_rng[2];
      const bool pack_now = a.Nr == 0 || Lr == a.Nr;
      if (!(pack_now && Lp >= a.cap)) {
        if (pack_now) {
          a.w_packed_len[b] = Lp + 1;
          if (a.Nr > 0) a.w_res_head[b] = (rh + 1) % a.Nr;
        } else {
          a.w_res_len[b] = Lr + 1;
        }
      }
    }
  };
  if (a.S == 1) {
    if (STEP && threadIdx.x == 0) commit_step(atomicInc(&a.seq_tickets[b], (unsigned)(a.Hkv - 1)));
    return;
  }
  // the last split of this KV head to finish merges all S partials
  if (take_last_ticket_acq_rel<NTHREADS>(a, bh, &s_last)) {
    // (the sequence ticket's round trip overlaps the combine)
    unsigned seq_ticket = 0;
    if (STEP && threadIdx.x == 0) seq_ticket = atomicInc(&a.seq_tickets[b], (unsigned)(a.Hkv - 1));
    const int i = warp, e = lane * 4;
    float* oacc = a.o_acc + (bh * QB + i) * D + e;
    // the flag and the accumulators in one round trip
    const uint32_t far = __ldcg(&a.fb_flag[bh]);
    const float4 o = __ldcg(reinterpret_cast<const float4*>(oacc));
    const float L = __ldcg(&a.l_acc[bh * QB + i]);
    if (far != 0u) {
      // some split's max was too far above the reference: log-sum-exp merge of
      // the S partials
      combine_unit<NTHREADS, D, 8>(a, b, h, 0, reinterpret_cast<float*>(smem));
    } else if (i < a.gq) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      store_out4(a, ((int64_t)b * a.Hq + h * a.gq + i) * D + e,
                 make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv));
    }
    // leave the head's accumulators, reference and flag at zero for the next call
    *reinterpret_cast<float4*>(oacc) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane == 0) {
      a.l_acc[bh * QB + i] = 0.f;
      a.ref_max[bh * QB + i] = 0u;
    }
    if (threadIdx.x == 0) a.fb_flag[bh] = 0u;
    commit_step(seq_ticket);
  }
}

// --------------------------------------------------------- tensor maps -----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's cuTensorMapEncodeTiled, looked up once per process.
EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// A 2D view [rows][row_bytes] of uint8 with a box of box_rows whole rows.
bool encode_rows_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows,
                     CUtensorMapSwizzle swz, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0 || rows > 0x7fffffffull) return false;  // y is a 32-bit coordinate
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)row_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded tensor maps, reused across calls.  A map is a pure function of its
// key (base address, row bytes, rows, swizzle, box), so an entry stays valid
// even after the memory behind it is freed and reallocated; a serving loop over
// the layers of a model finds all its caches here after its first step.  The
// table is emptied when it reaches kMapCacheMax entries.
struct RowsMapKey {
  const void* base;
  uint64_t row_bytes, rows;
  int swz;
  uint32_t box;
  bool operator==(const RowsMapKey& o) const {
    return base == o.base && row_bytes == o.row_bytes && rows == o.rows && swz == o.swz &&
           box == o.box;
  }
};
struct RowsMapKeyHash {
  size_t operator()(const RowsMapKey& k) const {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    h ^= (k.rows + 0x632BE59BD9B4E019ull * (k.row_bytes + 131 * (uint64_t)k.swz + 7919 * k.box)) +
         (h << 6) + (h >> 2);
    return (size_t)h;
  }
};
constexpr size_t kMapCacheMax = 4096;

bool make_rows_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows,
                   CUtensorMapSwizzle swz, uint32_t box_rows) {
  static std::mutex mu;
  static std::unordered_map<RowsMapKey, CUtensorMap, RowsMapKeyHash> cache;
  const RowsMapKey k = {base, row_bytes, rows, (int)swz, box_rows};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(k);
  if (it != cache.end()) {
    *map = it->second;
    return true;
  }
  if (!encode_rows_map(map, base, row_bytes, rows, swz, box_rows)) return false;
  if (cache.size() >= kMapCacheMax) cache.clear();
  cache.emplace(k, *map);
  return true;
}

// Raise the kernel's dynamic shared-memory limit once per device (the attribute
// is per device; a process may drive several GPUs).
template <int BITS, bool STEP, int CPS, int TT>
cudaError_t ensure_smem_attr(size_t smem) {
  static std::atomic<uint64_t> done{0};  // bit i: set on device i
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(decode_tc_kernel<BITS, STEP, CPS, TT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <int BITS, bool STEP, int CPS, int TT>
cudaError_t launch_bits(const Dims& s, const DecodePlan& p, const DecodeArgs& a, cudaStream_t st) {
  using Gm = Geo<BITS, CPS, TT>;
  // packed rows: every (sequence, head, slot), or every (page, head, slot) of a pool
  const bool paged = s.page != 0;
  if (paged && TT != 128) return cudaErrorInvalidValue;  // a warp's rows must be one page
  const uint64_t rows = paged ? (uint64_t)s.npages * s.Hkv * kPage : (uint64_t)s.B * s.Hkv * s.cap;
  const uint32_t box = paged ? kPage : Gm::T;
  CUtensorMap kc, vc;
  // INT3 rows (48 bytes) load unswizzled: each warp re-lays them out itself
  const CUtensorMapSwizzle swz = BITS == 4   ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : BITS == 3 ? CU_TENSOR_MAP_SWIZZLE_NONE
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
  if (!make_rows_map(&kc, a.k_codes, Gm::RB, rows, swz, box) ||
      !make_rows_map(&vc, a.v_codes, Gm::RB, rows, swz, box))
    return cudaErrorInvalidValue;
  constexpr size_t smem = tc_smem_bytes<BITS, CPS, TT>();
  cudaError_t e = ensure_smem_attr<BITS, STEP, CPS, TT>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.splits, (unsigned)s.Hkv, (unsigned)s.B);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<BITS, STEP, CPS, TT>, kc, vc, a);
}

}  // namespace

bool tc_supported(const kvq_cache_desc& D, int gq) {
  return D.head_dim == 128 && gq >= 1 && gq <= QB && D.capacity > 0 && encode_fn() != nullptr;
}

int tc_threads() { return NTHREADS; }
int tc_ctas_per_sm(bool several_waves) { return several_waves ? 4 : 3; }
int tc_residual_rows() { return kResRows; }
int tc_tile_tokens(const kvq_cache_desc& D, int cps, int64_t split_tokens) {
  // measured on INT2 only: 128K tokens (2,425 per split) 38.0 -> 37.0 us;
  // 32K tokens (604 per split) 14.5 -> 15.0 us, so short splits keep 128
  return D.bits == 2 && cps == 3 && D.page_size == 0 && split_tokens >= 8 * 192 ? 192 : 128;
}

template <int CPS>
cudaError_t launch_cps(const Dims& s, const DecodePlan& p, const DecodeArgs& a, cudaStream_t st,
                       bool step) {
  if (s.bits == 3)
    return step ? launch_bits<3, true, CPS, 128>(s, p, a, st) : launch_bits<3, false, CPS, 128>(s, p, a, st);
  if (s.bits == 4)
    return step ? launch_bits<4, true, CPS, 128>(s, p, a, st) : launch_bits<4, false, CPS, 128>(s, p, a, st);
  if (CPS == 3 && p.tile == 192)
    return step ? launch_bits<2, true, 3, 192>(s, p, a, st) : launch_bits<2, false, 3, 192>(s, p, a, st);
  return step ? launch_bits<2, true, CPS, 128>(s, p, a, st) : launch_bits<2, false, CPS, 128>(s, p, a, st);
}

cudaError_t launch_decode_tc(const Dims& s, const DecodePlan& p, const DecodeArgs& a,
                             cudaStream_t st, bool step) {
  return p.cps == 4 ? launch_cps<4>(s, p, a, st, step) : launch_cps<3>(s, p, a, st, step);
}

}  // namespace kvq
