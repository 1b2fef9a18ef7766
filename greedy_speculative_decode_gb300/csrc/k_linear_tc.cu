// k_linear_tc.cu -- the batch-invariant linear for blocks of 9 to 128 rows on
// the fifth-generation tensor cores (tcgen05): Y[m, n] = sum_k X[m, k] W[n, k].
//
// Same weight stream, split and epilogues as the mma.sync form, with the
// multiply moved off the consumer warps.  Each ring stage holds a 128-row x
// 64-column weight block and the 32 x 64 (or, for prefill blocks of more
// than 32 rows, 128 x 64) block of the input rows at the same columns (one
// TMA box; rows past M are never stored).  One thread issues, per block, four
// tcgen05.mma of 128 x N x 16 (weight rows as the 128-row operand, the token
// rows padded to N = 16, 32 or 128 as the N-column one) into an fp32
// accumulator in tensor memory; a tile piece (a CTA's run of k-blocks inside
// one 128-row tile) starts from zero, and two accumulators alternate so the
// next piece runs while the consumers read the last one back, 32 token rows
// at a time.
//
// Bit-identity with the mma.sync form (and so with single-token decode):
// every output element is the fp32 sum of the same products taken 16 k at a
// time in k order from zero, which the two instructions round identically
// (checked element by element on random, small-weight and wide-range
// operands); pieces and split partials are summed in the same order.
//
// Roles: warps 0-7 consumers (RMSNorm of each stage's input rows in place
// when the linear has a norm prologue, accumulator read-back, split-tile
// exchange, epilogues), warp 8 the TMA producer, warp 9 the MMA issuer.
// Every wait is bounded; on a timeout the kernel raises ST_TIMEOUT, waits
// (bounded) for its own copies and multiplies, and frees its tensor memory.
#include "lin_dev.cuh"
#include "linear_tc.h"

namespace sv {
namespace {

constexpr int kTcThreads = (kLinConsumerWarps + 2) * 32;
constexpr int kTcProducerWarp = kLinConsumerWarps, kTcMmaWarp = kLinConsumerWarps + 1;

// Geometry of the form for MP padded token rows (16, 32 or 128).
template <int MP>
struct TcGeom {
  static constexpr int kXRows = MP <= 32 ? 32 : MP;                   // rows of the input box
  static constexpr int kStageBytes = kLinStageBytes + kXRows * 128;  // weight block + input box
  static constexpr int kStages = MP <= 32 ? 8 : 6;
  static constexpr int kAcc = MP <= 32 ? 32 : MP;    // tensor-memory columns between the two accumulators
  static constexpr int kCols = MP <= 32 ? 64 : 256;  // tensor-memory columns allocated (a power of 2)
  static constexpr int kCR = MP <= 32 ? MP : 32;     // token rows per read-back / epilogue chunk
  static_assert(kStageBytes % 1024 == 0, "swizzle atoms stay aligned");
};

// ---------------------------------------------------------------- tcgen05
// Shared-memory operand descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the TMA box layout); start address >> 4 in bits 0-13,
// leading offset 1 (unused by swizzled K-major operands), stride 1024 >> 4 in
// bits 32-45, descriptor version 1 at bit 46, layout 2 (128B swizzle) at 61.
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major; N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accum)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Eight consecutive accumulator columns of the warp's 32 lanes.
__device__ __forceinline__ void tc_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- layout
struct TcSmem {
  uint8_t* ring;        // [S][weight 16 KB | input box]
  float* T;             // [128][kCR + 1] epilogue tile
  uint64_t* full;       // [S] the stage's weight and input bytes landed
  uint64_t* xnorm;      // [S] the stage's input rows are normalised (by one consumer warp)
  uint64_t* empty;      // [S] the multiplies reading the stage completed
  uint64_t* acc_full;   // [2] an accumulator holds a finished piece
  uint64_t* acc_empty;  // [2] the consumers read it back (8 consumer warps)
  uint64_t* drain;      // the issuer's last multiplies completed
  uint64_t* gbar;       // the gain window landed
  bf16* gs;             // [kLinXCols] gain of the CTA's input window (norm prologue)
  float* s_rstd;        // [MP]
  float* s_hrstd;       // [64]
  uint32_t* taddr;      // tensor-memory base address from tcgen05.alloc
};

template <int MP>
__device__ __forceinline__ TcSmem tc_smem(uint8_t* smem) {
  using G = TcGeom<MP>;
  TcSmem sm;
  sm.ring = smem;
  sm.T = reinterpret_cast<float*>(smem + G::kStages * G::kStageBytes);
  sm.full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sm.T) +
                                        ((kLinRows * (G::kCR + 1) * sizeof(float) + 15) & ~size_t(15)));
  sm.xnorm = sm.full + G::kStages;
  sm.empty = sm.xnorm + G::kStages;
  sm.acc_full = sm.empty + G::kStages;
  sm.acc_empty = sm.acc_full + 2;
  sm.drain = sm.acc_empty + 2;
  sm.gbar = sm.drain + 1;
  sm.gs = reinterpret_cast<bf16*>(sm.gbar + 1);
  sm.s_rstd = reinterpret_cast<float*>(sm.gs + kLinXCols);
  sm.s_hrstd = sm.s_rstd + MP;
  sm.taddr = reinterpret_cast<uint32_t*>(sm.s_hrstd + 64);
  return sm;
}

template <int MP>
constexpr size_t tc_smem_bytes() {
  using G = TcGeom<MP>;
  return 1024 /* alignment slack */ + (size_t)G::kStages * G::kStageBytes +
         (((size_t)kLinRows * (G::kCR + 1) * sizeof(float) + 15) & ~size_t(15)) +
         (3 * G::kStages + 6) * sizeof(uint64_t) + kLinXCols * sizeof(bf16) + (MP + 64) * sizeof(float) + 16;
}
static_assert(tc_smem_bytes<128>() <= 232448, "fits the per-block shared-memory limit");

// ---------------------------------------------------------------- producer
// One thread.  The weight boxes of the first S blocks go out before the wait
// on the previous kernel (weights never depend on it), their input boxes
// after it; then both for each block as its stage frees up.  Returns the
// number of blocks issued through `issued` and false on a timeout.
template <int MP>
__device__ bool tc_produce(const LinParams& p, const CUtensorMap* wmap, const CUtensorMap* xmap, int cta,
                           int G, const TcSmem& sm, long long& issued) {
  constexpr int S = TcGeom<MP>::kStages, SB = TcGeom<MP>::kStageBytes;
  const int KB = p.Kd / kLinBK;
  long long kb_begin, kb_end;
  lin_range(p, cta, G, kb_begin, kb_end);
  const long long n = kb_end - kb_begin;
  const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
  issued = 0;
  if (n <= 0) return true;
  int tile = (int)(kb_begin / KB), kk = (int)(kb_begin % KB);
  auto weight = [&](int s) {
    load_weight_block(p, wmap, sm.ring + s * SB, tile, kk, &sm.full[s], pol_w);
  };
  auto input = [&](int s, int kcol) {
    tma_load_2d(sm.ring + s * SB + kLinStageBytes, xmap, kcol * kLinBK, 0, &sm.full[s], pol_x);
  };
  auto advance = [&]() {
    if (++kk == KB) {
      kk = 0;
      ++tile;
    }
  };
  const int pre = (int)(n < S ? n : S);
  const int kk_first = kk;
  for (int s = 0; s < pre; ++s) {
    mbar_arrive_expect_tx(&sm.full[s], SB);
    weight(s);
    advance();
  }
  pdl_wait();  // the input rows come from the previous kernel
  for (int s = 0, kc = kk_first; s < pre; ++s) {
    input(s, kc);
    if (++kc == KB) kc = 0;
  }
  issued = pre;
  for (long long i = pre; i < n; ++i) {
    const int s = (int)(i % S);
    if (!mbar_wait(&sm.empty[s], (uint32_t)((i / S) & 1) ^ 1u)) return false;
    mbar_arrive_expect_tx(&sm.full[s], SB);
    weight(s);
    input(s, kk);
    advance();
    issued = i + 1;
  }
  return true;
}

// Wait (bounded) until the copies of the last use of every stage landed.
template <int MP>
__device__ void tc_produce_drain(const TcSmem& sm, long long issued) {
  constexpr int S = TcGeom<MP>::kStages;
  for (long long u = issued - 1; u >= 0 && u >= issued - S; --u) mbar_wait(&sm.full[u % S], (uint32_t)((u / S) & 1));
}

// ---------------------------------------------------------------- MMA issuer
// One thread: per block, wait for its bytes (and, with a norm prologue, for
// the normalised input rows), then four k16 multiplies; the stage is released
// when they complete, the accumulator when the piece's last ones complete.
template <bool NORM, int MP>
__device__ bool tc_issue(const LinParams& p, int cta, int G, const TcSmem& sm, uint32_t tmem) {
  const int KB = p.Kd / kLinBK;
  long long kb_begin, kb_end;
  lin_range(p, cta, G, kb_begin, kb_end);
  constexpr uint32_t idesc = tc_idesc(kLinRows, MP);
  constexpr int S = TcGeom<MP>::kStages, SB = TcGeom<MP>::kStageBytes;
  long long left = kb_end - kb_begin;
  int kk0 = (int)(kb_begin % KB);
  long long it = 0;
  int piece = 0;
  bool ok = true;
  while (left > 0 && ok) {
    const int nblk = (int)(left < KB - kk0 ? left : KB - kk0);
    const int b = piece & 1;
    if (piece >= 2 && !mbar_wait(&sm.acc_empty[b], (uint32_t)((piece / 2) & 1) ^ 1u)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem + (uint32_t)(b * TcGeom<MP>::kAcc);
    for (int j = 0; j < nblk; ++j, ++it) {
      const int s = (int)(it % S);
      const uint32_t par = (uint32_t)((it / S) & 1);
      if (!mbar_wait(&sm.full[s], par)) {
        ok = false;
        break;
      }
      if (NORM && !mbar_wait(&sm.xnorm[s], par)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a_base = smem_u32(sm.ring + s * SB), b_base = a_base + kLinStageBytes;
#pragma unroll
      for (int k16 = 0; k16 < kLinBK / 16; ++k16)
        tc_mma(d_tmem, tc_sdesc(a_base + 32 * k16), tc_sdesc(b_base + 32 * k16), idesc, j > 0 || k16 > 0);
      tc_commit(&sm.empty[s]);
    }
    if (!ok) break;
    tc_commit(&sm.acc_full[b]);
    ++piece;
    left -= nblk;
    kk0 = 0;
  }
  // every multiply this thread issued has completed before tensor memory is freed
  tc_commit(sm.drain);
  if (!mbar_wait(sm.drain, 0)) ok = false;
  return ok;
}

// ---------------------------------------------------------------- consumers
// Split-tile exchange.  A CTA's partial slot holds 128 x 128 fp32 words,
// token rows in quads and tile rows innermost: the quad (c .. c + 3), c a
// multiple of 4, of tile row lr is at words 4 (32 c + lr) .. + 3, so a warp
// (32 consecutive tile rows) stores and polls 512 contiguous bytes per
// instruction.  A word not yet written holds kTcEmpty, a NaN with the sign
// bit set: arithmetic only produces the canonical NaN 0x7fffffff, so no
// partial sum is ever equal to it.  Quads of padding rows (c >= M) are not
// exchanged.  The reducer puts kTcEmpty back into every word it consumed.
constexpr uint32_t kTcEmpty = 0xffffffffu;

__device__ __forceinline__ uint32_t* tc_quad(uint32_t* slot, int lr, int c) { return slot + 4 * (32 * c + lr); }

__device__ __forceinline__ void st_relaxed_v4_u32(uint32_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void ld_relaxed_v4_u32(const uint32_t* p, uint4& v) {
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
}

// Split-tile reducer: v holds this CTA's piece (segment 0) of the CW values
// at tile row lr, token rows mb .. mb + CW - 1; add the partials that CTAs
// cta + 1 ... cta + nseg - 1 left in their slots, in segment order, sixteen
// quads (four segments of 32 rows, eight of 16) per polling round.  Returns
// false if a partial never arrived.
template <int CW>
__device__ __forceinline__ bool tc_gather(uint32_t* slots, int cta, int nseg, int lr, int mb, int M,
                                          float (&v)[CW]) {
  constexpr int QS = CW / 4, NQ = 16, B = NQ / QS;  // quad i: segment j0 + i / QS, rows mb + 4 (i mod QS) ..
  bool ok = true;
  for (int j0 = 1; j0 < nseg; j0 += B) {
    auto addr = [&](int i) {
      return tc_quad(slots + (size_t)(cta + j0 + i / QS) * kLinRows * kTcMaxRows, lr, mb + 4 * (i % QS));
    };
    uint4 x[NQ];
    uint32_t live = 0;
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      x[i] = make_uint4(0u, 0u, 0u, 0u);
      if (j0 + i / QS < nseg && mb + 4 * (i % QS) < M) {
        live |= 1u << i;
        ld_relaxed_v4_u32(addr(i), x[i]);
      }
    }
    auto missing = [&]() {
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < NQ; ++i)
        if (((live >> i) & 1u) &&
            (x[i].x == kTcEmpty || x[i].y == kTcEmpty || x[i].z == kTcEmpty || x[i].w == kTcEmpty))
          m |= 1u << i;
      return m;
    };
    uint32_t m = missing();
    if (m != 0) {
      const unsigned long long t0 = globaltimer_ns();
      for (;;) {
#pragma unroll
        for (int i = 0; i < NQ; ++i)
          if ((m >> i) & 1u) ld_relaxed_v4_u32(addr(i), x[i]);
        m = missing();
        if (m == 0) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      if ((live >> i) & 1u) {
        const int c = 4 * (i % QS);
        v[c] = __fadd_rn(v[c], __uint_as_float(x[i].x));
        v[c + 1] = __fadd_rn(v[c + 1], __uint_as_float(x[i].y));
        v[c + 2] = __fadd_rn(v[c + 2], __uint_as_float(x[i].z));
        v[c + 3] = __fadd_rn(v[c + 3], __uint_as_float(x[i].w));
        st_relaxed_v4_u32(addr(i), kTcEmpty, kTcEmpty, kTcEmpty, kTcEmpty);
      }
    }
  }
  return ok;
}

// Row rstd of the input from the per-128-column partial sums of squares, in
// the mma.sync form's order (lane-strided sums, then an xor tree); warp w
// takes rows w + 8 k, all four rows' loads in flight together.
template <int MP>
__device__ __forceinline__ void tc_row_rstd(const LinParams& p, const TcSmem& sm, int warp, int lane) {
  constexpr int R = MP / kLinConsumerWarps;
  float ss[R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int m = warp + kLinConsumerWarps * k;
    ss[k] = 0.0f;
    if (m < p.M)
      for (int t = lane; t < p.ss_tiles; t += 32) ss[k] = __fadd_rn(ss[k], __ldcg(p.x_ss + m * p.ss_tiles + t));
  }
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int m = warp + kLinConsumerWarps * k;
    for (int o = 16; o > 0; o >>= 1) ss[k] = __fadd_rn(ss[k], __shfl_xor_sync(0xffffffffu, ss[k], o));
    if (lane == 0 && m < p.M) sm.s_rstd[m] = 1.0f / sqrtf(ss[k] / (float)p.Kd + p.eps);
  }
}

template <int EPI, bool NORM, int MP>
__device__ bool tc_consume(const LinParams& p, uint32_t* slots, int cta, int G, const TcSmem& sm, uint32_t tmem) {
  using Geo = TcGeom<MP>;
  constexpr int S = Geo::kStages, SB = Geo::kStageBytes;
  constexpr int CR = Geo::kCR, TS = CR + 1, CW = CR / 2;  // chunk rows; CW: a warp's token rows of a chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nthr = kLinConsumerWarps * 32;
  const int KB = p.Kd / kLinBK;
  const long long Tk = (long long)p.n_tiles * KB;
  long long kb_begin, kb_end;
  lin_range(p, cta, G, kb_begin, kb_end);
  if (kb_begin >= kb_end) return true;
  // The gain of the input window (columns c0 + t mod Kd, t < ncols) does not
  // depend on earlier kernels: staged before the wait when it fits.
  int c0 = 0, ncols = 0;
  lin_window(p, kb_begin, kb_end, c0, ncols);
  const bool gain_staged = NORM && ncols <= kLinXCols;
  if (gain_staged && tid == 0) {
    const int first = min(ncols, p.Kd - c0);
    mbar_arrive_expect_tx(sm.gbar, (uint32_t)(ncols * sizeof(bf16)));
    bulk_load(sm.gs, p.gain + c0, (uint32_t)(first * sizeof(bf16)), sm.gbar);
    if (first < ncols) bulk_load(sm.gs + first, p.gain, (uint32_t)((ncols - first) * sizeof(bf16)), sm.gbar);
  }
  pdl_wait();  // sums of squares, the step state and the residual come from earlier kernels
  int pos = 0, cap = 0;
  if (EPI == EPI_QKV) {
    pos = __ldcg(&p.st->step_pos);
    cap = __ldcg(&p.st->cap_len);
  }
  bool ok = true;
  if (NORM) {
    tc_row_rstd<MP>(p, sm, warp, lane);
    if (gain_staged && !mbar_wait(sm.gbar, 0)) ok = false;
    named_sync(1, nthr);
  }
  // accumulator read-back, CR token rows (one chunk) at a time: warp w owns
  // tensor-memory lanes (tile rows) 32 (w mod 4) + lane and the chunk's token
  // rows mb .. mb + CW - 1
  const int lr = 32 * (warp & 3) + lane, mb = CW * (warp >> 2);
  const int nch = (p.M + CR - 1) / CR;  // chunks that hold rows
  float* T = sm.T;
  EpiPre<CR> pre;
  long long it = 0;
  int piece = 0;
  int tile = (int)(kb_begin / KB), kk0 = (int)(kb_begin % KB);
  long long left = kb_end - kb_begin;
  while (left > 0) {
    const int nblk = (int)(left < KB - kk0 ? left : KB - kk0);
    if (NORM) {
      // block `it` is normalised by consumer warp it mod S, so S blocks are
      // in hand at once and every use of a stage has the same owner (waits
      // on a stage's barrier then never run two phases ahead, where the
      // parity would alias); lane l takes the 16-byte chunk l mod 8 of rows
      // 4 i + l / 8 (four rows of 128 contiguous bytes per access: no bank
      // conflicts).  128B swizzle: chunk pc of row m holds columns
      // 8 (pc ^ (m mod 8)) .. + 7 of the block.
      static_assert(S <= kLinConsumerWarps, "a consumer warp per stage");
      for (int j = 0; j < nblk; ++j, ++it) {
        if ((int)(it % S) != warp) continue;
        const int s = (int)(it % S);
        if (ok && !mbar_wait(&sm.full[s], (uint32_t)((it / S) & 1))) ok = false;
        if (ok) {
          uint8_t* xb = sm.ring + s * SB + kLinStageBytes;
          const int pc = lane & 7;
          int wc = (kk0 + j) * kLinBK - c0;  // window column of the block
          if (wc < 0) wc += p.Kd;
          const uint4* g = gain_staged ? reinterpret_cast<const uint4*>(sm.gs + wc)
                                       : reinterpret_cast<const uint4*>(p.gain + (kk0 + j) * kLinBK);
#pragma unroll 4
          for (int i = 0; i < MP / 4; ++i) {
            const int m = 4 * i + (lane >> 3);
            if (m < p.M) {
              uint4* ptr = reinterpret_cast<uint4*>(xb + m * 128 + pc * 16);
              const int gc = pc ^ (m & 7);
              *ptr = norm8(*ptr, sm.s_rstd[m], gain_staged ? g[gc] : __ldg(g + gc));
            }
          }
        }
        fence_proxy_async_smem();  // the multiplies read these rows through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.xnorm[s]);
      }
    }
    // ------------ this CTA's piece of the tile is complete (k-blocks kk0 .. kk0 + nblk - 1)
    const int kk = kk0 + nblk - 1, kk_first = kk0, tile_done = tile;
    left -= nblk;
    ++tile;
    kk0 = 0;
    const int b = piece & 1;
    if (ok && !mbar_wait(&sm.acc_full[b], (uint32_t)((piece / 2) & 1))) ok = false;
    tc_fence_after();
    ++piece;
    const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(b * Geo::kAcc + mb);
    for (int ch = 0; ch < nch; ++ch) {
      const int r0 = ch * CR;  // first token row of the chunk
      float v[CW];
      if (ok) {
#pragma unroll
        for (int c = 0; c < CW; c += 8) tc_ld8(ta + r0 + c, v + c);
      } else {
#pragma unroll
        for (int c = 0; c < CW; ++c) v[c] = 0.0f;
      }
      if (ch == nch - 1) {  // the accumulator is free once its last chunk is in registers
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[b]);
      }
      if (kk_first != 0) {
        // A later segment of a split tile (the first piece of this CTA's
        // range): leave the partial in this CTA's slot and move on.
        uint32_t* slot = slots + (size_t)cta * kLinRows * kTcMaxRows;
#pragma unroll
        for (int c = 0; c < CW; c += 4)
          if (r0 + mb + c < p.M)
            st_relaxed_v4_u32(tc_quad(slot, lr, r0 + mb + c), __float_as_uint(v[c]), __float_as_uint(v[c + 1]),
                              __float_as_uint(v[c + 2]), __float_as_uint(v[c + 3]));
        continue;
      }
      // The chunk's rows r0 .. r0 + CR - 1 as an epilogue of up to CR rows:
      // the same epilogue code, its row pointers and positions moved by r0.
      LinParams pc = p;
      if (MP > CR) {
        pc.M = min(CR, p.M - r0);
        pc.out = p.out + (size_t)r0 * p.out_stride;
        if (EPI == EPI_RESID) pc.out_ss = p.out_ss + (size_t)r0 * p.n_tiles;
      }
      const int pos_c = pos + r0;
      epi_preload<CR, EPI>(pc, tile_done, pos_c, cap, pre);
      if (kk != KB - 1) {
        // The first segment of a split tile (the last piece of this CTA's
        // range): add the later segments' partials in k order.
        const int nseg = owner_cta((long long)tile_done * KB + KB - 1, Tk, G) - cta + 1;
        if (!tc_gather<CW>(slots, cta, nseg, lr, r0 + mb, p.M, v)) ok = false;
      }
      named_sync(1, nthr);  // the previous epilogue is done with T
#pragma unroll
      for (int c = 0; c < CW; ++c) T[lr * TS + mb + c] = v[c];
      named_sync(1, nthr);
      if (EPI == EPI_QKV)
        epilogue_qkv<CR>(pc, tile_done, T, TS, sm.s_hrstd, pos_c, pre);
      else if (EPI == EPI_RESID)
        epilogue_resid<CR>(pc, tile_done, T, TS, pre);
      else if (EPI == EPI_GLU)
        epilogue_glu(pc, tile_done, T, TS);
      else
        epilogue_logits<CR>(pc, tile_done, T, TS);
    }
  }
  return ok;
}

// Persistent stream-K linear, same partition as k_linear (one CTA per SM,
// equal contiguous k-block ranges, split tiles finished by their first CTA).
template <int EPI, bool NORM, int MP>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_linear_tc(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap pfmap,
                const __grid_constant__ CUtensorMap xmap, const LinParams p, uint32_t* slots) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  using Geo = TcGeom<MP>;
  const TcSmem sm = tc_smem<MP>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < Geo::kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.xnorm[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], kLinConsumerWarps);
    }
    mbar_init(sm.drain, 1);
    mbar_init(sm.gbar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {  // one warp allocates (and later frees) the two accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sm.taddr)),
                 "n"(Geo::kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.taddr;
  pdl_trigger();  // the next kernel may start its own weight stream
  bool ok = true;
  if (warp == kTcProducerWarp) {
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      prefetch_tensormap(&xmap);
      long long issued = 0;
      ok = tc_produce<MP>(p, &wmap, &xmap, blockIdx.x, gridDim.x, sm, issued);
      if (ok) lin_prefetch_next(p, &pfmap, blockIdx.x);
      tc_produce_drain<MP>(sm, issued);
    }
  } else if (warp == kTcMmaWarp) {
    if (lane == 0) ok = tc_issue<NORM, MP>(p, blockIdx.x, gridDim.x, sm, tmem);
  } else {
    ok = tc_consume<EPI, NORM, MP>(p, slots, blockIdx.x, gridDim.x, sm, tmem);
  }
  if (!ok && lane == 0) atomicOr(&p.st->status, ST_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(Geo::kCols)
                 : "memory");
  }
}

template <int EPI, bool NORM, int MP>
cudaError_t launch_tc_t(const LinearDesc& d, const CUtensorMap& xmap, uint32_t* slots, const LinParams& p,
                        cudaStream_t s, bool pdl, const CUtensorMap& pfmap) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d.grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = tc_smem_bytes<MP>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_linear_tc<EPI, NORM, MP>, d.map, pfmap, xmap, p, slots);
}

// RMS-normalised input rows for the tcgen05 form (steps of more than 8
// rows): xn[m, :] = bf16(bf16(x[m, :] rstd_m) gain), rstd_m from the
// per-128-column sums of squares in tc_row_rstd's order (lane-strided sums,
// then an xor tree), so xn holds exactly the values the norm prologue would
// write (into every ring stage, for 128-row blocks), once per linear instead
// of once per CTA or weight tile.  Block (c, m): row m, 16-byte
// vectors c * 256 + threadIdx.x, ...
__global__ void __launch_bounds__(256) k_norm_rows(const bf16* __restrict__ x, const float* __restrict__ x_ss,
                                                   const bf16* __restrict__ gain, bf16* __restrict__ xn, int H,
                                                   int ss_tiles, float eps) {
  pdl_trigger();
  pdl_wait();  // x and its sums of squares come from the previous kernel
  const int m = blockIdx.y;
  __shared__ float s_r;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float ss = 0.0f;
    for (int t = lane; t < ss_tiles; t += 32) ss = __fadd_rn(ss, __ldcg(x_ss + m * ss_tiles + t));
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (lane == 0) s_r = 1.0f / sqrtf(ss / (float)H + eps);
  }
  __syncthreads();
  const float r = s_r;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)m * H);
  uint4* yr = reinterpret_cast<uint4*>(xn + (size_t)m * H);
  for (int c8 = blockIdx.x * blockDim.x + threadIdx.x; c8 < H / 8; c8 += gridDim.x * blockDim.x)
    yr[c8] = norm8(__ldcg(xr + c8), r, __ldg(reinterpret_cast<const uint4*>(gain) + c8));
  asm volatile("fence.proxy.async.global;" ::: "memory");  // read next through TMA
}

template <int EPI, bool NORM, int MP>
cudaError_t prepare_tc_mp() {
  return cudaFuncSetAttribute(k_linear_tc<EPI, NORM, MP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tc_smem_bytes<MP>());
}

template <int EPI, bool NORM>
cudaError_t prepare_tc_t() {
  cudaError_t e;
  if ((e = prepare_tc_mp<EPI, NORM, 16>()) != cudaSuccess) return e;
  if ((e = prepare_tc_mp<EPI, NORM, 32>()) != cudaSuccess) return e;
  if constexpr (EPI == EPI_LOGITS) {  // the LM head runs on at most 32 rows
    if ((e = prepare_tc_mp<EPI, false, 16>()) != cudaSuccess) return e;
    return prepare_tc_mp<EPI, false, 32>();
  } else {
    if constexpr (NORM) {  // the step's rows may come normalised by k_norm_rows
      if ((e = prepare_tc_mp<EPI, false, 128>()) != cudaSuccess) return e;
      if ((e = prepare_tc_mp<EPI, false, 16>()) != cudaSuccess) return e;
      if ((e = prepare_tc_mp<EPI, false, 32>()) != cudaSuccess) return e;
    }
    return prepare_tc_mp<EPI, NORM, 128>();
  }
}

template <int MP>
cudaError_t launch_tc_mp(const LinearDesc& d, const CUtensorMap& xmap, uint32_t* slots, const LinParams& p,
                         int epi, bool norm, cudaStream_t s, bool pdl, const CUtensorMap& pf) {
  switch (epi) {
    case EPI_QKV:
      // (rows normalised by k_norm_rows, or here in the prologue)
      return norm ? launch_tc_t<EPI_QKV, true, MP>(d, xmap, slots, p, s, pdl, pf)
                  : launch_tc_t<EPI_QKV, false, MP>(d, xmap, slots, p, s, pdl, pf);
    case EPI_RESID:
      return norm ? cudaErrorInvalidValue : launch_tc_t<EPI_RESID, false, MP>(d, xmap, slots, p, s, pdl, pf);
    case EPI_GLU:
      return norm ? launch_tc_t<EPI_GLU, true, MP>(d, xmap, slots, p, s, pdl, pf)
                  : launch_tc_t<EPI_GLU, false, MP>(d, xmap, slots, p, s, pdl, pf);
    case EPI_LOGITS:  // the LM head runs on at most 32 rows
      if (MP > 32) return cudaErrorInvalidValue;
      return norm ? launch_tc_t<EPI_LOGITS, true, (MP > 32 ? 32 : MP)>(d, xmap, slots, p, s, pdl, pf)
                  : launch_tc_t<EPI_LOGITS, false, (MP > 32 ? 32 : MP)>(d, xmap, slots, p, s, pdl, pf);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_norm_rows(const bf16* x, const float* x_ss, const bf16* gain, bf16* xn, int M, int H,
                             float eps, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((H / 8 + 255) / 256, M);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_norm_rows, x, x_ss, gain, xn, H, H / 128, eps);
}

size_t linear_tc_smem_bytes(int mp) {
  return mp <= 16 ? tc_smem_bytes<16>() : (mp <= 32 ? tc_smem_bytes<32>() : tc_smem_bytes<128>());
}

cudaError_t prepare_linear_tc_kernels() {
  cudaError_t e;
  if ((e = prepare_tc_t<EPI_QKV, true>()) != cudaSuccess) return e;
  if ((e = prepare_tc_t<EPI_RESID, false>()) != cudaSuccess) return e;
  if ((e = prepare_tc_t<EPI_GLU, true>()) != cudaSuccess) return e;
  return prepare_tc_t<EPI_LOGITS, true>();
}

cudaError_t launch_linear_tc(const LinearDesc& d, const CUtensorMap& xmap, uint32_t* slots, const LinParams& p_in,
                             int epi, bool norm, cudaStream_t s, bool pdl, const LinearDesc* next) {
  if (p_in.M < 1 || p_in.M > kTcMaxRows) return cudaErrorInvalidValue;
  LinParams p = p_in;
  if (next) {
    p.pf_blocks = kLinPrefetchBlocks;
    p.pf_n_tiles = next->n_tiles;
    p.pf_Kd = next->Kd;
    p.pf_grid = next->grid;
    p.pf_map = next->map_kind;
    p.pf_ffn = next->N / 2;  // gate|up: the up rows start at ffn
    p.pf_wt = next->tiled;
  } else {
    p.pf_blocks = 0;
    p.pf_wt = nullptr;
  }
  const CUtensorMap& pf = next ? next->map : d.map;
  if (p.M <= 16) return launch_tc_mp<16>(d, xmap, slots, p, epi, norm, s, pdl, pf);
  if (p.M <= 32) return launch_tc_mp<32>(d, xmap, slots, p, epi, norm, s, pdl, pf);
  return launch_tc_mp<128>(d, xmap, slots, p, epi, norm, s, pdl, pf);
}

}  // namespace sv
