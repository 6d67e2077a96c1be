// Step 4 of the method (summary page of "Block Sparse Attention with Log-Linear
// Complexity", section "Method step details", step 4; section "Prerequisites", BSA:
// attention on the raw K/V of the selected blocks only).  The softmax runs over the
// connected positions only (blog post of the same title, section 3.3): for query t and
// head h, the keys of the selected blocks of h's group, restricted to keys <= t.
//
// The G_Q heads of one query share the selected blocks, so one warp owns one query: its
// G_Q rows (padded to 16) form the M = 16 side of m16n8k16 MMAs; different queries
// select different blocks, so there is no larger dense tile without wasted work.  The
// kernel is bound by moving the selected K/V blocks into the SM.  Each warp of a CTA (12
// warps at d = 128, 16 at d = 64) runs its own ring of shared-memory slots (2 at d = 128,
// 3 at d = 64) filled by TMA (one 4-D box per 32-key half block: rows x both 64-column
// halves of d, 128-byte swizzle, rows past N read as zero); the ring keeps the next loads in
// flight while the current slot is multiplied, across block and query boundaries, and
// skips half blocks that hold no visible key.
// S = Q K^T and O += P V use ldmatrix (.trans for V) on the swizzled slots; the softmax is
// online in the exp2 domain against a lazy reference maximum per row: exact on the first half
// block, then moved (and O and the running sum rescaled) only when a logit passes it by more
// than 2^8, so most half blocks need no cross-lane maximum and no rescale.  Keys are masked
// only in half blocks that reach past the last visible key.
// All waits are bounded.
#include "kernels.cuh"

namespace pisa {
namespace {

// Warps per CTA (one query each) and ring slots per warp.  The kernel is latency-bound, so
// it runs as many warps as the register file holds, with the rest of shared memory as ring.
constexpr int nw_for(int d) { return d == 128 ? 12 : 16; }
constexpr int nslot_for(int d) { return d == 128 ? 2 : 3; }
constexpr int KS = 32;      // keys per slot (half a block)
constexpr float RESCALE_MARGIN = 8.f;  // exp2 headroom before O and l are rescaled (P <= 2^8)

struct AttnParams {
  const uint16_t* Q;
  const int32_t* idx;
  uint16_t* O;
  float* LSE;
  long long total;  // B * H_kv * (queries in [t_lo, t_hi))
  int BH;           // B * H_kv
  int N, H_q, H_kv, GQ, Ksel, M1, causal;
  int t_lo, nq;     // queries t_lo .. t_lo + nq - 1 are attended
  int one_box;      // 1: the 4-D map loads both d halves in one box
  float sl2;     // softmax scale x log2(e)
  float margin;  // RESCALE_MARGIN / sl2: headroom of the reference maximum in raw logit units
};

// Walks the (query, selected block, half block, K|V) load sequence of one warp.  Items are
// (bh, t) pairs, t in [t_lo, t_lo + nq), visited with a grid stride; the stride is applied
// as (bh, t) increments.
struct Cursor {
  int bh, t;        // current item; bh >= BH when exhausted
  unsigned mask;    // remaining valid idx positions of the item
  int val;          // this lane's idx entry of the item
  int blk, nsub, sub, kv;
};

struct Stride {
  int bh, t;     // the grid stride in items, as (bh, t) increments
  int t_end, nq;  // the query range ends at t_end and holds nq queries
};

__device__ __forceinline__ void step_item(int& bh, int& t, const Stride& st) {
  t += st.t;
  bh += st.bh;
  if (t >= st.t_end) {
    t -= st.nq;
    ++bh;
  }
}

__device__ __forceinline__ int half_blocks(const AttnParams& p, int blk, int t) {
  const int last = p.causal ? min(t, p.N - 1) : p.N - 1;
  int cnt = last - blk * 64 + 1;
  if (cnt > 64) cnt = 64;
  return (cnt + KS - 1) / KS;
}

__device__ __forceinline__ void first_block(Cursor& c, const AttnParams& p) {
  c.sub = 0;
  c.kv = 0;
  if (c.mask) {
    c.blk = __shfl_sync(0xffffffffu, c.val, __ffs(c.mask) - 1);
    c.nsub = half_blocks(p, c.blk, c.t);
  }
}

// Loads the selection row of item (c.bh, c.t) into the cursor.
__device__ __forceinline__ void load_item(Cursor& c, const AttnParams& p, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  c.val = -1;
  c.mask = 0;
  if (c.bh >= p.BH) return;
  const long long item = (long long)c.bh * p.N + c.t;
  int v = lane < p.Ksel ? p.idx[item * p.Ksel + lane] : -1;
  if (v >= p.M1) {
    report_error(err, ERR_BAD_INDEX);
    v = -1;
  }
  // a block that starts after t has no visible key: skip it
  if (v >= 0 && p.causal && v * 64 > c.t) v = -1;
  c.val = v;
  c.mask = __ballot_sync(0xffffffffu, v >= 0);
  first_block(c, p);
}

template <int D, int NW = nw_for(D), int NSLOT = nslot_for(D)>
__global__ void __launch_bounds__(32 * NW, 1) sparse_attn_kernel(const __grid_constant__ CUtensorMap mapK,
                                                                 const __grid_constant__ CUtensorMap mapV,
                                                                 AttnParams p, uint32_t* err) {
  constexpr int HALVES = D / 64;
  constexpr uint32_t SLOT = KS * D * 2;
  constexpr uint32_t HALF = KS * 128;  // bytes of one 64-column half of a slot
  constexpr int KST = D / 16;          // k-steps of Q K^T
  constexpr int NDT = D / 8;           // n-tiles of P V
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[NW][NSLOT];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, q = lane & 3;
  uint8_t* ring = smem + (size_t)warp * NSLOT * SLOT;
  // per-lane byte offsets of the ldmatrix rows inside a 128-byte-swizzled slot (16-byte
  // chunk c of key row k sits at chunk c ^ (k & 7)): K fragments at d chunk lane/8 (+4 for
  // odd 32-column groups), V fragments at key lane%16 and d chunk 2j + lane/16; every
  // address below is one of these plus a compile-time constant
  const uint32_t llo = lane & 7;
  const uint32_t koff0 = llo * 128 + ((((uint32_t)lane >> 3) ^ llo) << 4);
  const uint32_t koff1 = llo * 128 + (((4u ^ ((uint32_t)lane >> 3)) ^ llo) << 4);
  uint32_t voff[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    voff[j] = ((((uint32_t)lane >> 3) & 1u) * 8 + llo) * 128 + (((2u * j) ^ ((uint32_t)lane >> 4) ^ llo) << 4);
  if (lane == 0) {
    for (int i = 0; i < NSLOT; ++i) mbar_init(&full[warp][i], 1);
    mbar_fence_init();
  }
  __syncwarp();

  // K/V blocks are re-read by many queries: keep them in L2; Q and O stream through once
  const uint64_t keep_policy = l2_evict_last_policy();
  const uint64_t stream_policy = l2_evict_first_policy();
  const long long gw = (long long)blockIdx.x * NW + warp;
  const long long nwarps = (long long)gridDim.x * NW;
  const Stride st{(int)(nwarps / p.nq), (int)(nwarps % p.nq), p.t_lo + p.nq, p.nq};
  const int bh0 = (int)(gw / p.nq), t0 = p.t_lo + (int)(gw % p.nq);

  // ---- producer side of this warp's ring ----
  Cursor pc;
  pc.bh = bh0;
  pc.t = t0;
  load_item(pc, p, err);
  while (pc.mask == 0 && pc.bh < p.BH) {
    step_item(pc.bh, pc.t, st);
    load_item(pc, p, err);
  }
  // ring state: loads in flight, next slot to fill, next slot to consume and its parity
  int in_flight = 0, islot = 0, cslot = 0;
  uint32_t cphase = 0;
  auto issue_fill = [&]() {
    while (in_flight < NSLOT && pc.bh < p.BH) {
      const int slot = islot;
      const int bh = pc.bh;
      const int row = pc.blk * 64 + pc.sub * KS;
      // the slot's previous contents were read by ldmatrix whose results fed MMAs issued
      // before this point, so the reads are complete when the copy is issued
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[warp][slot], SLOT);
        const CUtensorMap* m = pc.kv == 0 ? &mapK : &mapV;
        uint8_t* dst = ring + slot * SLOT;
        if (p.one_box) {
          tma_load_4d_hint(dst, m, &full[warp][slot], 0, row, 0, bh, keep_policy);
        } else {
#pragma unroll
          for (int h = 0; h < HALVES; ++h) tma_load_3d_hint(dst + h * HALF, m, &full[warp][slot], 64 * h, row, bh, keep_policy);
        }
      }
      islot = islot + 1 == NSLOT ? 0 : islot + 1;
      ++in_flight;
      // advance: K then V of each half block, half blocks of each block, blocks of each item
      pc.kv ^= 1;
      if (pc.kv == 0 && ++pc.sub == pc.nsub) {
        pc.mask &= pc.mask - 1;
        first_block(pc, p);
        while (pc.mask == 0 && pc.bh < p.BH) {
          step_item(pc.bh, pc.t, st);
          load_item(pc, p, err);
        }
      }
    }
  };
  issue_fill();
  auto consume_next = [&]() {
    if (++cslot == NSLOT) {
      cslot = 0;
      cphase ^= 1u;
    }
    --in_flight;
  };

  bool ok = true;
  for (int bh = bh0, t = t0; bh < p.BH && ok; step_item(bh, t, st)) {
    const int b = bh / p.H_kv, hk = bh - b * p.H_kv;
    Cursor cc;
    cc.bh = bh;
    cc.t = t;
    load_item(cc, p, nullptr);
    {  // move the next item's selection row and Q rows towards L2 while this one runs
      int nbh = bh, nt = t;
      step_item(nbh, nt, st);
      if (nbh < p.BH) {
        const long long nitem = (long long)nbh * p.N + nt;
        const int nb = nbh / p.H_kv, nhk = nbh - nb * p.H_kv;
        const uint16_t* nq = p.Q + (((size_t)nb * p.N + nt) * p.H_q + (size_t)nhk * p.GQ) * D;
        if (lane * 64 < p.GQ * D) prefetch_l2(nq + (size_t)lane * 64);  // 128 bytes per lane
        if (lane == 31) prefetch_l2(p.idx + nitem * p.Ksel);
      }
    }

    // Q fragments (rows r, r+8 of the group; zero past G_Q)
    uint32_t qa[KST][4];
    const uint16_t* qrow = p.Q + (((size_t)b * p.N + t) * p.H_q + (size_t)hk * p.GQ) * D;
#pragma unroll
    for (int ks = 0; ks < KST; ++ks) {
      const int c0 = 16 * ks + 2 * q;
      qa[ks][0] = r < p.GQ ? ld_b32_hint(qrow + (size_t)r * D + c0, stream_policy) : 0u;
      qa[ks][1] = r + 8 < p.GQ ? ld_b32_hint(qrow + (size_t)(r + 8) * D + c0, stream_policy) : 0u;
      qa[ks][2] = r < p.GQ ? ld_b32_hint(qrow + (size_t)r * D + c0 + 8, stream_policy) : 0u;
      qa[ks][3] = r + 8 < p.GQ ? ld_b32_hint(qrow + (size_t)(r + 8) * D + c0 + 8, stream_policy) : 0u;
    }
    float o[NDT][4];
#pragma unroll
    for (int i = 0; i < NDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // m0/m1: reference row maxima in raw logit units (exact after the first half block, then
    // raised only when a logit passes them by more than RESCALE_MARGIN in the exp2 domain)
    float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
    float th0 = NEG_INF, th1 = NEG_INF;  // rescale thresholds m + margin / sl2
    const int last = p.causal ? min(t, p.N - 1) : p.N - 1;  // last visible key

    while (cc.mask && ok) {
      const int kbase = cc.blk * 64 + cc.sub * KS;
      // ---------------- S = Q K^T over KS keys ----------------
      if (!mbar_wait_warp(&full[warp][cslot], cphase, err)) {
        ok = false;
        break;
      }
      const uint32_t kb = smem_u32(ring + cslot * SLOT);
      // even and odd k-steps accumulate separately (s, s2) and are added at the end: two
      // chains of four dependent MMAs per n-tile instead of one of eight, so the warp waits
      // less on the MMA latency
      float s[KS / 8][4], s2[KS / 8][4];
#pragma unroll
      for (int nt = 0; nt < KS / 8; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[nt][c] = s2[nt][c] = 0.f;
      // per 32 columns of d: all n-tiles' fragments first, then two rounds of independent MMAs
#pragma unroll
      for (int kp = 0; kp < KST / 2; ++kp) {
        uint32_t bk[KS / 8][4];
#pragma unroll
        for (int nt = 0; nt < KS / 8; ++nt) {
          const uint32_t addr = kb + ((kp & 1) ? koff1 : koff0) + (kp >> 1) * HALF + nt * 1024;
          ldmatrix_x4(addr, bk[nt][0], bk[nt][1], bk[nt][2], bk[nt][3]);
        }
#pragma unroll
        for (int nt = 0; nt < KS / 8; ++nt)
          mma_bf16_16816(s[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], bk[nt][0], bk[nt][1]);
#pragma unroll
        for (int nt = 0; nt < KS / 8; ++nt)
          mma_bf16_16816(s2[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2], qa[2 * kp + 1][3], bk[nt][2],
                         bk[nt][3]);
      }
#pragma unroll
      for (int nt = 0; nt < KS / 8; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[nt][c] += s2[nt][c];
      consume_next();
      issue_fill();

      // ---------------- online softmax (exp2 domain, lazy reference maximum) ----------------
      if (kbase + KS - 1 > last) {  // the half block holds invisible keys: mask them
#pragma unroll
        for (int nt = 0; nt < KS / 8; ++nt) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const bool vis = kbase + 8 * nt + 2 * q + c <= last;
            s[nt][c] = vis ? s[nt][c] : NEG_INF;
            s[nt][2 + c] = vis ? s[nt][2 + c] : NEG_INF;
          }
        }
      }
      // this lane's row maxima of the half block, then one test against the thresholds
      float mx0 = fmaxf(s[0][0], s[0][1]), mx1 = fmaxf(s[0][2], s[0][3]);
#pragma unroll
      for (int nt = 1; nt < KS / 8; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      if (__any_sync(0xffffffffu, (mx0 > th0) | (mx1 > th1))) {
        // exact row maxima of this half block; move the reference and rescale O and l
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
        const float c0 = (nm0 == NEG_INF || nm0 == m0) ? 1.f : fast_exp2((m0 - nm0) * p.sl2);
        const float c1 = (nm1 == NEG_INF || nm1 == m1) ? 1.f : fast_exp2((m1 - nm1) * p.sl2);
        m0 = nm0;
        m1 = nm1;
        th0 = m0 + p.margin;
        th1 = m1 + p.margin;
        l0 *= c0;
        l1 *= c1;
#pragma unroll
        for (int i = 0; i < NDT; ++i) {
          o[i][0] *= c0;
          o[i][1] *= c0;
          o[i][2] *= c1;
          o[i][3] *= c1;
        }
      }
      // every processed half block holds a visible key, so m0 and m1 are finite here
      const float ms0 = -m0 * p.sl2, ms1 = -m1 * p.sl2;
      // exponent arguments and row sums two lanes per instruction (packed fp32)
      const unsigned long long sl2x2 = pack_f32x2(p.sl2, p.sl2);
      const unsigned long long ms0x2 = pack_f32x2(ms0, ms0), ms1x2 = pack_f32x2(ms1, ms1);
      unsigned long long lx0 = 0ull, lx1 = 0ull;
      uint32_t pa[KS / 16][4];
#pragma unroll
      for (int nt = 0; nt < KS / 8; ++nt) {
        float x00, x01, x10, x11;
        unpack_f32x2(fma_f32x2(pack_f32x2(s[nt][0], s[nt][1]), sl2x2, ms0x2), x00, x01);
        unpack_f32x2(fma_f32x2(pack_f32x2(s[nt][2], s[nt][3]), sl2x2, ms1x2), x10, x11);
        const float p00 = fast_exp2(x00), p01 = fast_exp2(x01);
        const float p10 = fast_exp2(x10), p11 = fast_exp2(x11);
        lx0 = add_f32x2(lx0, pack_f32x2(p00, p01));
        lx1 = add_f32x2(lx1, pack_f32x2(p10, p11));
        const int kk = nt >> 1, hi = nt & 1;
        pa[kk][hi ? 2 : 0] = pack_bf16x2(p00, p01);
        pa[kk][hi ? 3 : 1] = pack_bf16x2(p10, p11);
      }

      {
        float a0, b0, a1, b1;
        unpack_f32x2(lx0, a0, b0);
        unpack_f32x2(lx1, a1, b1);
        l0 += a0 + b0;
        l1 += a1 + b1;
      }
      // ---------------- O += P V ----------------
      if (!mbar_wait_warp(&full[warp][cslot], cphase, err)) {
        ok = false;
        break;
      }
      const uint32_t vb = smem_u32(ring + cslot * SLOT);
#pragma unroll
      for (int kk = 0; kk < KS / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < NDT / 2; ++np) {
          const uint32_t addr = vb + voff[np & 3] + (np >> 2) * HALF + kk * 2048;
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(addr, b0, b1, b2, b3);
          mma_bf16_16816(o[2 * np], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
          mma_bf16_16816(o[2 * np + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
        }
      }
      consume_next();
      issue_fill();
      // next half block / block
      if (++cc.sub == cc.nsub) {
        cc.mask &= cc.mask - 1;
        first_block(cc, p);
      }
    }
    if (!ok) break;

    // ---------------- normalise and store ----------------
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    uint16_t* orow = p.O + (((size_t)b * p.N + t) * p.H_q + (size_t)hk * p.GQ) * D;
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      const int col = 8 * i + 2 * q;
      if (r < p.GQ) st_b32_hint(orow + (size_t)r * D + col, pack_bf16x2(o[i][0] * inv0, o[i][1] * inv0), stream_policy);
      if (r + 8 < p.GQ)
        st_b32_hint(orow + (size_t)(r + 8) * D + col, pack_bf16x2(o[i][2] * inv1, o[i][3] * inv1), stream_policy);
    }
    if (p.LSE && q == 0) {
      const size_t hbase = (size_t)b * p.H_q + (size_t)hk * p.GQ;
      if (r < p.GQ) p.LSE[(hbase + r) * p.N + t] = l0 > 0.f ? (m0 * p.sl2 + fast_log2(l0)) * LN2 : NEG_INF;
      if (r + 8 < p.GQ) p.LSE[(hbase + r + 8) * p.N + t] = l1 > 0.f ? (m1 * p.sl2 + fast_log2(l1)) * LN2 : NEG_INF;
    }
  }
  // drain loads still in flight before the CTA's shared memory goes away (bounded)
  while (in_flight > 0) {
    if (!mbar_wait_warp(&full[warp][cslot], cphase, err)) break;
    consume_next();
  }
}

template <int D>
cudaError_t launch_d(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx, uint16_t* O,
                     float* LSE, const Problem& p, int num_sms, uint32_t* err, cudaStream_t s) {
  constexpr int HALVES = D / 64;
  CUtensorMap mapK, mapV;
  AttnParams prm;
  // one box per half block: dims (64 columns, rows, d half, b*h_kv); the d-half dimension is
  // outermost in shared memory, giving two consecutive 128-byte-swizzled tiles
  {
    const uint64_t dims[4] = {64, (uint64_t)p.N, (uint64_t)HALVES, (uint64_t)p.B * p.H_kv};
    const uint64_t strides[3] = {(uint64_t)D * 2, 128, (uint64_t)p.N_cap * D * 2};
    const uint32_t box[4] = {64, (uint32_t)KS, (uint32_t)HALVES, 1};
    prm.one_box = encode_tensor_map(&mapK, K, 4, dims, strides, box) && encode_tensor_map(&mapV, V, 4, dims, strides, box);
  }
  if (!prm.one_box) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.N, (uint64_t)p.B * p.H_kv};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.N_cap * D * 2};
    const uint32_t box[3] = {64, (uint32_t)KS, 1};
    if (!encode_tensor_map(&mapK, K, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_tensor_map(&mapV, V, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  prm.Q = Q;
  prm.idx = idx;
  prm.O = O;
  prm.LSE = LSE;
  prm.t_lo = p.t_lo;
  prm.nq = p.t_hi - p.t_lo;
  prm.total = prm.nq > 0 ? (long long)p.B * p.H_kv * prm.nq : 0;
  prm.BH = p.B * p.H_kv;
  prm.N = p.N;
  prm.H_q = p.H_q;
  prm.H_kv = p.H_kv;
  prm.GQ = p.GQ;
  prm.Ksel = p.K;
  prm.M1 = (p.N + 63) / 64;
  prm.causal = p.causal;
  prm.sl2 = p.scale * LOG2E;
  prm.margin = RESCALE_MARGIN / prm.sl2;
  if (prm.total == 0) return cudaSuccess;
  constexpr int NW = nw_for(D), NSLOT = nslot_for(D);
  const size_t smem = (size_t)NW * NSLOT * KS * D * 2 + 1024;
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  long long blocks = (prm.total + NW - 1) / NW;
  if (blocks > num_sms) blocks = num_sms;
  sparse_attn_kernel<D><<<(int)blocks, 32 * NW, smem, s>>>(mapK, mapV, prm, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_attn(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                               uint16_t* O, float* LSE, const Problem& p, int num_sms, uint32_t* err, cudaStream_t s) {
  if (p.d == 128) return launch_d<128>(Q, K, V, idx, O, LSE, p, num_sms, err, s);
  return launch_d<64>(Q, K, V, idx, O, LSE, p, num_sms, err, s);
}

}  // namespace pisa
