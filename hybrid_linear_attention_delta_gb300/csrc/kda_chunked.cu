// kda_chunked.cu -- chunked KDA prefill on tcgen05 tensor cores (sm_103a).
//
// The recurrence (gated delta rule with per-channel decay; "Kimi K3 on vLLM:
// Up to 370 Tokens/sec", section "Kimi Delta Attention: a hybrid recurrent +
// full-attention stack") is evaluated in chunks of C = 64 tokens.  For a chunk
// with start state S0 (dk x dv) and in-chunk cumulative log-decay G_r (per
// channel), the state after each token unrolls to
//     S_r = Diag(e^{G_r}) S0 + sum_{i<=r} Diag(e^{G_r - G_i}) k_i u_i^T,
// and the write vectors u_r solve a unit lower-triangular system (the WY / UT
// transform):
//     (I + A) U = Diag(beta) (V - K+ S0),  A = Diag(beta) strict_lower(K+ K-^T)
//     T = (I + A)^{-1} Diag(beta),  W = T K+,  U = T V - W S0
//     O = Q+ S0 + lower_incl(Q+ K-^T) U
//     S_end = Diag(e^{G_C}) S0 + (K * e^{G_C - G})^T U
// with K+ = K e^{G}, K- = K e^{-G}, Q+ = Q e^{G} (per channel).
//
// Exponents are anchored at the chunk midpoint a = G_32 (the cumulative decay
// after row 31): K+ = K e^{G - a}, K- = K e^{a - G} and Q+ = Q e^{G - a} keep
// |G - a| within half a chunk's decay; the anchor cancels in K+ K-^T and
// Q+ K-^T and is folded into the bf16 copy of the start state,
// S0' = Diag(e^{a}) S0, so W S0 and Q+ S0 use S0'.
//
// One CTA (8 warps) owns one (sequence, head, dv block) and walks its chunks
// in order; the fp32 state lives in registers (thread = one state row, half of
// the block's columns).  Per chunk:
//   TMA   q, k, v, g tiles (128-byte swizzled) into one of two stages
//         (the next chunk's tiles load while this one computes)
//   prep  cumulative decay per channel, K+, Q+, K- (in place), S0'
//   MMA1  [K+; Q+] K-^T                 M=128 N=64  K=128  -> A, Q+K-^T (TMEM)
//   solve T = (I + A)^{-1} Diag(beta)    fp32, 32x32 blocks, CUDA cores
//         (an idle solve thread requests the next chunk's tiles)
//   MMA2  [T; M] K+ and [T; M] V        -> W, U~ (TMEM)
//   MMA3  U~ -= W S0'  (O = Q+ S0' was issued before the solve)
//   MMA4  K-^T U       ;  O += M U
//   out   o rows -> smem -> TMA store; S = Diag(e^{G_C}) S + Diag(e^{G_C - a}) K-^T U
//         (= K_end^T U with K_end = K e^{G_C - G}) in registers; a snapshot
//         -> the chunk's own (dead) input stage -> fp32 TMA store (dense
//         buffer or retained pool slot); the final state -> global fp32
// Below it, the cooperative mode for few (sequence, head) pairs splits the same
// chunk pipeline between producer CTAs and one state-carrying CTA per pair.
// All MMAs are M = 128 (rows 64..127 of the 64-row operands are ignored).
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = 64;
constexpr int kDK = 128;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;

template <int DV>
struct Layout {
  // one input stage: [k h0 | q h0 | k h1 | q h1] (8 KiB each; K+ / Q+ in place),
  // v halves, g halves (K- in place, then solve scratch)
  static constexpr uint32_t kQ = 8192;
  static constexpr uint32_t kV = 32768;
  static constexpr uint32_t kG = kV + (DV / 64) * 8192;
  static constexpr uint32_t kStage = kG + 16384;
  static constexpr uint32_t kTM = 2 * kStage;          // [T; M]: 128 rows x 64 tokens
  static constexpr uint32_t kW = kTM + 16384;          // W halves
  static constexpr uint32_t kU = kW + 16384;           // U halves; X_00^T, A_10 during the solve
  static constexpr uint32_t kScr = kU + 16384;         // solve scratch (16 KiB)
  static constexpr uint32_t kS0 = kScr + 16384;        // S0' halves (128 rows each)
  static constexpr uint32_t kMisc = kS0 + (DV / 64) * 16384;
  static constexpr uint32_t kBars = 0;                 // tma[2], mma
  static constexpr uint32_t kSlot = 24;                // TMEM base address
  static constexpr uint32_t kBeta = 64;                // f32[64]
  static constexpr uint32_t kTot = kBeta + 256;        // f32[128] G_C (chunk decay)
  static constexpr uint32_t kAnc = kTot + 512;         // f32[128] a (anchor decay)
  static constexpr uint32_t kEa = kAnc + 512;          // f32[128] e^{a} (cooperative producer)
  static constexpr uint32_t kCke = kEa + 512;          // f32[128] e^{G_C} (cooperative producer)
  static constexpr uint32_t kSeqs = kCke + 512;        // int2[64] (tok0, len) per sequence
  static constexpr uint32_t kBytes = kMisc + kSeqs + 512;
  // prep scratch: per 4-row group decay sums f32[16][128], in the T rows of
  // [T; M] (8 KiB; the solve rewrites them and zeroes T's upper blocks)
  static constexpr uint32_t kGpart = kTM;
  // solve scratch (fp32): X_00^T (rows 0..31 of 64 read by its product) and
  // A_10 in the U buffer; X_11, Y^T (X_11's padding rows) and the transposed
  // diagonal blocks of A in kScr
  static constexpr uint32_t kXd = kScr;                 // f32[32][32]
  static constexpr uint32_t kYt = kScr + 4096;          // f32[32][32]
  static constexpr uint32_t kLT = kScr + 8192;          // f32[2][32][32]
  static_assert(kStage % 1024 == 0, "stage alignment");
  static_assert(kBytes <= 232448, "shared memory budget");
};

struct ChunkArgs {
  const __nv_bfloat16 *beta;
  const SeqMeta *meta;
  const int32_t *order;
  float *pool;
  __nv_bfloat16 *out;
  float *snaps;
  const int32_t *snap_slots;  // retention map, or NULL (dense snapshots)
  int64_t snaps_capacity;
  int32_t snap_interval;
  int32_t H, dv, n_dvb;
  uint32_t *err;
  // [B*H] by (longest-first rank * H + head): set to epoch for a unit whose
  // decay left the chunked algorithm's exponent range; such a unit's final
  // state is not written here (its source stays intact) and the exact
  // token-recurrent kernel recomputes it after this kernel
  uint32_t *rerun;
  uint32_t epoch;
  // per-state kernel: snapshots leave through TMA stores (fp32 maps over the
  // snapshot buffer and the pool are valid); else through direct stores
  int32_t snap_tma;
};

// A CTA-uniform bounded wait: false (for every thread) if any thread gave up.
__device__ __forceinline__ bool cta_wait(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return !__syncthreads_or(!ok);
}

__device__ __forceinline__ void st_bf(uint8_t *base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(x);
}

// A 32-column fp32 matrix stored by rows of 8 float4 chunks, chunk c of row r
// at position c ^ (r & 7): the 128-byte swizzled K-major layout of a tf32
// tensor-core operand (rows that differ in their low bits hit different banks).
__device__ __forceinline__ int sidx(int r, int i) {
  return r * 32 + ((((i >> 2) ^ (r & 7)) << 2) | (i & 3));
}

// T = (I + A)^{-1} Diag(beta) for the 64x64 strictly lower A.  X = (I + A)^{-1}
// is built from 32 x 32 blocks:
//  * the diagonal blocks X_00, X_11 by forward substitution, warps 0-3 on
//    X_00 and warps 4-7 on X_11, each column shared by four lanes of a warp
//    (rows 0..7, 8..15, 16..23, 24..31);
//  * the block below them, X_10 = -X_11 (A_10 X_00), as two 32 x 32 x 32
//    products on the tensor cores in tf32 (fp32 accumulation; the operands'
//    11-bit significands keep their rounding under the bf16 rounding T then
//    takes): Y^T = X_00^T A_10^T, then X_10 = -X_11 Y, each 4 MMAs of M = 64
//    (rows 32..63 of A are padding whose results are not read) into TMEM
//    columns [0, 32) and [32, 64), which no chunk phase holds during the solve.
// Operands, fp32 rows of 32 in the 128-byte swizzled K-major layout (sidx):
// X_00^T at XT (64 rows read, 32 written), A_10 at A10 (written by
// extract_am), X_11 at Xd followed by Y^T at YT (X_11's padding rows are
// Y^T's).  LT holds the two diagonal blocks of A transposed (LT[b][m][i] =
// A[32b + i][32b + m], written by extract_am), so the substitution runs column
// by column: once x[m] is known it is folded into the running sums of every
// later row, and x[m + 1] is one multiply-add away.  T is written as bf16
// into rows 0..63 of the K-major [T; M] operand at tm, whose upper block
// threads 0..127 first zero (the rows also hold the decay prefix scratch of
// the chunk's preparation) after running side(tid), brief work of the caller
// that does not touch the solve's buffers.  bar / phase: the
// chunk's MMA barrier and the parity of its next completion (advanced twice).
// Ends with T fenced for the tensor cores and a barrier; false when a wait
// gave up (pending then says whether an MMA is still in flight).
template <class Side>
__device__ __forceinline__ bool solve_T(const float *LT, float *XT, const float *A10, float *Xd,
                                        float *YT, const float *beta, uint8_t *tm, uint32_t tmem,
                                        uint32_t bar, uint32_t &phase, bool &pending, int tid,
                                        const Side &side) {
  fence_async_smem();  // A10 (extract_am) for the tensor cores
  if (tid < 128) {  // T's upper block: rows 0..31, 16-byte chunks 4..7
    side(tid);
    *reinterpret_cast<uint4 *>(tm + sw128_chunk(tid >> 2, 4 + (tid & 3))) = make_uint4(0, 0, 0, 0);
  }
  {
    // warp w: block b = w / 4, columns j = 8 (w % 4) .. +7 of it (lane % 8);
    // lane / 8 picks the column's rows 8 (lane / 8) .. +7
    const int lane = tid & 31, w = tid >> 5, b = w >> 2, rq = lane >> 3;
    const int j = 8 * (w & 3) + (lane & 7), base = 32 * b, r0 = 8 * rq;
    const float *lt = LT + b * 1024 + r0;
    float t[8], xo[8];  // running sums and values of this lane's rows r0 + e
#pragma unroll
    for (int e = 0; e < 8; ++e) t[e] = 0.f;
    auto sel = [&](int m, float v) { return m < j ? 0.f : (m == j ? 1.f : v); };
#pragma unroll
    for (int g = 0; g < 8; ++g) {  // columns m0 .. m0 + 3, owned by the lanes of rows quarter g / 2
      const int m0 = 4 * g;
      float l[4][8];  // column m0 + k of A at this lane's rows
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float4 v = *reinterpret_cast<const float4 *>(lt + (m0 + k) * 32 + 4 * q);
          l[k][4 * q] = v.x;
          l[k][4 * q + 1] = v.y;
          l[k][4 * q + 2] = v.z;
          l[k][4 * q + 3] = v.w;
        }
      // the 4 x 4 triangle, on every lane (meaningful on the owner of rows m0..m0+3)
      const int e0 = m0 & 7;
      const float y0 = sel(m0, t[e0]);
      const float y1 = sel(m0 + 1, fmaf(-l[0][e0 + 1], y0, t[e0 + 1]));
      const float y2 = sel(m0 + 2, fmaf(-l[1][e0 + 2], y1, fmaf(-l[0][e0 + 2], y0, t[e0 + 2])));
      const float y3 =
          sel(m0 + 3, fmaf(-l[2][e0 + 3], y2,
                           fmaf(-l[1][e0 + 3], y1, fmaf(-l[0][e0 + 3], y0, t[e0 + 3]))));
      const int src = (lane & 7) + 8 * (g >> 1);
      const float x0 = __shfl_sync(0xffffffffu, y0, src), x1 = __shfl_sync(0xffffffffu, y1, src);
      const float x2 = __shfl_sync(0xffffffffu, y2, src), x3 = __shfl_sync(0xffffffffu, y3, src);
      if (rq == (g >> 1)) {
        xo[e0] = x0;
        xo[e0 + 1] = x1;
        xo[e0 + 2] = x2;
        xo[e0 + 3] = x3;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e)  // columns m0.. of A are zero at rows <= their index
        t[e] = fmaf(-l[3][e], x3, fmaf(-l[2][e], x2, fmaf(-l[1][e], x1, fmaf(-l[0][e], x0, t[e]))));
    }
    const float bj = beta[base + j];
    if (b == 0) {  // row j of X_00^T: entries r0 .. r0 + 7
#pragma unroll
      for (int q = 0; q < 2; ++q)
        *reinterpret_cast<float4 *>(XT + sidx(j, r0 + 4 * q)) =
            make_float4(xo[4 * q], xo[4 * q + 1], xo[4 * q + 2], xo[4 * q + 3]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) Xd[sidx(r0 + e, j)] = xo[e];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) st_bf(tm, sw128_offset(base + r0 + e, base + j), xo[e] * bj);
  }
  fence_async_smem();  // X_00^T, X_11 for the tensor cores
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t xt = smem_u32(XT), a10 = smem_u32(A10), xd = smem_u32(Xd), yt = smem_u32(YT);
  if (tid == 0) {  // Y^T = X_00^T A_10^T
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_tf32(tmem, sw128_desc(xt + kk * 32, 16, 1024), sw128_desc(a10 + kk * 32, 16, 1024),
               idesc_tf32(64, 32), kk > 0);
    mma_commit(bar);
  }
  pending = true;
  if (!cta_wait(bar, phase)) return false;
  phase ^= 1;
  pending = false;
  tc_fence_after();
  if (warp < 2) {  // M = 64 rows 0..31 sit in lanes 0..15 of quarters 0 and 1
    float v[32];
    tmem_ld32(lane_base, v);
    if (lane < 16) {
      const int jr = 16 * warp + lane;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4 *>(YT + sidx(jr, 4 * q)) =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {  // X_10 = -X_11 Y
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_tf32(tmem + 32, sw128_desc(xd + kk * 32, 16, 1024), sw128_desc(yt + kk * 32, 16, 1024),
               idesc_tf32(64, 32, 1), kk > 0);
    mma_commit(bar);
  }
  pending = true;
  if (!cta_wait(bar, phase)) return false;
  phase ^= 1;
  pending = false;
  tc_fence_after();
  if (warp < 2) {  // rows 32 + i of T, columns 0..31: X_10 Diag(beta)
    float v[32];
    tmem_ld32(lane_base + 32, v);
    if (lane < 16) {
      const int i = 16 * warp + lane;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float *bc = beta + 8 * c;
        *reinterpret_cast<uint4 *>(tm + sw128_chunk(32 + i, c)) =
            make_uint4(pack_bf16x2(v[8 * c] * bc[0], v[8 * c + 1] * bc[1]),
                       pack_bf16x2(v[8 * c + 2] * bc[2], v[8 * c + 3] * bc[3]),
                       pack_bf16x2(v[8 * c + 4] * bc[4], v[8 * c + 5] * bc[5]),
                       pack_bf16x2(v[8 * c + 6] * bc[6], v[8 * c + 7] * bc[7]));
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  return true;
}

// ------------------------------------------------------------------ chunk phases
// The steps of one chunk that do not depend on its start state, shared by the
// single-CTA kernel and the producer role of the cooperative kernel.  Ly is
// the shared-memory layout; VCOLS the v columns staged per chunk.

// Decay-scaled operands of one chunk, in place in its stage: K+ over k, Q+
// over q, K- over g; per channel the anchor a (s_anc) and the chunk decay G_C
// (s_tot); beta (s_beta, from beta_r of threads 0..63, which load_beta
// fetched before the chunk's tiles landed); v rows past a ragged end zeroed.
// Thread: channels [8 cq, 8 cq + 8) x rows [4 rg, 4 rg + 4), 16-byte accesses.
// Ends with the operand writes fenced for the tensor cores and a barrier.
// A channel whose decay within one half of the chunk exceeds kMaxHalfDecay
// nats would overflow e^{|G - a|} in fp32 / bf16: the function then returns
// true (on every thread), and the caller hands the whole (sequence, head) to
// the token-recurrent kernel, which has no such limit.
constexpr float kMaxHalfDecay = 80.f;

// beta of row tid of a chunk (threads 0..63; zero past the chunk's end), read
// early so that its global-memory latency overlaps the wait for the tiles
__device__ __forceinline__ float load_beta(const __nv_bfloat16 *beta_t0, int H, int cl, int tid) {
  return tid < cl ? __bfloat162float(beta_t0[(int64_t)tid * H]) : 0.f;
}

template <class Ly, int VCOLS>
__device__ __forceinline__ bool prep_chunk(uint32_t sb, int cl, float beta_r, float *s_gpart,
                                           float *s_beta, float *s_tot, float *s_anc, int tid) {
  const int cq = tid & 15, rg = tid >> 4;
  const uint32_t okq = (cq >> 3) * 16384, og = Ly::kG + (cq >> 3) * 8192;
  float gl[4][8];  // in-group inclusive cumulative decay
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int r = 4 * rg + rr;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (r < cl) w = ld_shared_v4(sb + og + sw128_chunk(r, cq & 7));
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      gl[rr][2 * j] = (rr ? gl[rr - 1][2 * j] : 0.f) + bf16lo(wv[j]);
      gl[rr][2 * j + 1] = (rr ? gl[rr - 1][2 * j + 1] : 0.f) + bf16hi(wv[j]);
    }
  }
  float4 *gp = reinterpret_cast<float4 *>(s_gpart + rg * 128 + 8 * cq);
  gp[0] = make_float4(gl[3][0], gl[3][1], gl[3][2], gl[3][3]);
  gp[1] = make_float4(gl[3][4], gl[3][5], gl[3][6], gl[3][7]);
  if (tid < 64) s_beta[tid] = beta_r;
  if (cl < kC) {  // ragged tail: zero the v rows past the sequence end
    for (int e = tid; e < (kC - cl) * (VCOLS / 8); e += kThreads) {
      const int r = cl + e / (VCOLS / 8), chk = e % (VCOLS / 8);
      st_shared_v4(sb + Ly::kV + (chk >> 3) * 8192 + sw128_chunk(r, chk & 7), 0, 0, 0, 0);
    }
  }
  __syncthreads();
  if (tid < 128) {  // per channel: exclusive prefix over the 16 row groups (in place)
    float run = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < 16; ++g2) {
      const float p = s_gpart[g2 * 128 + tid];
      s_gpart[g2 * 128 + tid] = run;
      run += p;
      if (g2 == 7) s_anc[tid] = run;  // a: decay through row 31
    }
    s_tot[tid] = run;                  // G_C: decay through the chunk
  }
  __syncthreads();
  // (G - a) log2(e) before this thread's rows: each scale factor is then one
  // base-2 exponential of a multiply-add
  constexpr float kLog2e = 1.44269504088896341f;
  float pre[8];
  {
    const float4 *pp = reinterpret_cast<const float4 *>(s_gpart + rg * 128 + 8 * cq);
    const float4 *pa = reinterpret_cast<const float4 *>(s_anc + 8 * cq);
    const float4 p0 = pp[0], p1 = pp[1], a0 = pa[0], a1 = pa[1];
    pre[0] = (p0.x - a0.x) * kLog2e; pre[1] = (p0.y - a0.y) * kLog2e;
    pre[2] = (p0.z - a0.z) * kLog2e; pre[3] = (p0.w - a0.w) * kLog2e;
    pre[4] = (p1.x - a1.x) * kLog2e; pre[5] = (p1.y - a1.y) * kLog2e;
    pre[6] = (p1.z - a1.z) * kLog2e; pre[7] = (p1.w - a1.w) * kLog2e;
  }
  float xmax = 0.f;  // largest |G_r - a| log2(e) of the chunk's rows
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int r = 4 * rg + rr;
    const uint32_t ck = sw128_chunk(r, cq & 7);
    uint32_t kp[4] = {0, 0, 0, 0}, qp[4] = {0, 0, 0, 0}, km[4] = {0, 0, 0, 0};
    if (r < cl) {
      const uint4 kw = ld_shared_v4(sb + okq + ck);
      const uint4 qw = ld_shared_v4(sb + Ly::kQ + okq + ck);
      const uint32_t kv[4] = {kw.x, kw.y, kw.z, kw.w}, qv[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x0 = fmaf(gl[rr][2 * j], kLog2e, pre[2 * j]);  // (G_r - a) log2(e)
        const float x1 = fmaf(gl[rr][2 * j + 1], kLog2e, pre[2 * j + 1]);
        xmax = fmaxf(xmax, fmaxf(fabsf(x0), fabsf(x1)));
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
        const float f0 = ex2_approx(-x0), f1 = ex2_approx(-x1);
        const float k0 = bf16lo(kv[j]), k1 = bf16hi(kv[j]);
        const float q0 = bf16lo(qv[j]), q1 = bf16hi(qv[j]);
        kp[j] = pack_bf16x2(k0 * e0, k1 * e1);
        qp[j] = pack_bf16x2(q0 * e0, q1 * e1);
        km[j] = pack_bf16x2(k0 * f0, k1 * f1);
      }
    }
    st_shared_v4(sb + okq + ck, kp[0], kp[1], kp[2], kp[3]);
    st_shared_v4(sb + Ly::kQ + okq + ck, qp[0], qp[1], qp[2], qp[3]);
    st_shared_v4(sb + og + ck, km[0], km[1], km[2], km[3]);
  }
  fence_async_smem();
  return __syncthreads_or(xmax > kMaxHalfDecay * kLog2e) != 0;
}

// MMA1: [K+; Q+] K-^T -> d (64 columns: rows 0..63 A-raw, rows 64..127 Q+K-^T).
template <class Ly>
__device__ __forceinline__ void issue_mma1(uint32_t d, uint32_t sb) {
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_bf16(d, sw128_desc(sb + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
             sw128_desc(sb + Ly::kG + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
             idesc_bf16(128, 64, 0, 0), kk > 0);
}

// A = Diag(beta) strict_lower(rows 0..63 of the MMA1 result at taddr): its
// two diagonal 32 x 32 blocks transposed into LT (LT[b][m][i] = A[32b + i][32b
// + m]) and the block below them, A_10, as fp32 rows of 32 in the 128-byte
// swizzled K-major layout at A10 (the solve's tensor-core operand); M =
// lower_incl(Q+ K-^T) (rows 64..127) as bf16 into rows 64..127 of [T; M] at tm.
__device__ __forceinline__ void extract_am(uint32_t taddr, int quarter, int colhalf, int lane,
                                           const float *s_beta, float *A10, float *LT, uint32_t tm) {
  const int rr = quarter * 32 + lane;
  if (quarter < 2) {
    if (quarter < colhalf) return;  // above the diagonal blocks: zero, not needed
    float v[32];
    tmem_ld32(taddr + colhalf * 32, v);
    const float br = s_beta[rr];
    float a[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) a[e] = colhalf * 32 + e < rr ? br * v[e] : 0.f;
    if (quarter == colhalf) {  // a diagonal block: lane = row within it
#pragma unroll
      for (int e = 0; e < 32; ++e) LT[quarter * 1024 + e * 32 + lane] = a[e];
    } else {  // A_10: row lane
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        *reinterpret_cast<float4 *>(A10 + sidx(lane, 4 * q4)) =
            make_float4(a[q4 * 4], a[q4 * 4 + 1], a[q4 * 4 + 2], a[q4 * 4 + 3]);
    }
  } else {
    float v[32];
    tmem_ld32(taddr + colhalf * 32, v);
    const int r = rr - 64;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float w8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = colhalf * 32 + q4 * 8 + j;
        w8[j] = (i <= r) ? v[q4 * 8 + j] : 0.f;
      }
      st_shared_v4(tm + sw128_chunk(64 + r, colhalf * 4 + q4), pack_bf16x2(w8[0], w8[1]),
                   pack_bf16x2(w8[2], w8[3]), pack_bf16x2(w8[4], w8[5]), pack_bf16x2(w8[6], w8[7]));
    }
  }
}

// MMA2: [T; M] K+ -> tmem[0, 128) and [T; M] V -> tmem[128, 128 + VCOLS).
template <class Ly, int VCOLS>
__device__ __forceinline__ void issue_mma2(uint32_t tmem, uint32_t tm, uint32_t sb) {
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint64_t ad = sw128_desc(tm + kk * 32, 16, 1024);
    mma_bf16(tmem + 0, ad, sw128_desc(sb + kk * 2048, 16384, 1024), idesc_bf16(128, 128, 0, 1),
             kk > 0);
    mma_bf16(tmem + 128, ad, sw128_desc(sb + Ly::kV + kk * 2048, 8192, 1024),
             idesc_bf16(128, VCOLS, 0, 1), kk > 0);
  }
}

// The cooperative producer's MMA2: W = [T; M] K+ -> tmem[0, 128) (rows 0..63)
// and U~^T = V^T T^T -> tmem[128, 192): TMEM lane = value column, TMEM
// column = token (V as an MN-major A operand with M = 128 value columns, T
// as the K-major B operand, N = K = 64 tokens), so that the package can carry
// U~ transposed, one 128-byte row per value column.
template <class Ly>
__device__ __forceinline__ void issue_mma2_coop(uint32_t tmem, uint32_t tm, uint32_t sb) {
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint64_t td = sw128_desc(tm + kk * 32, 16, 1024);
    mma_bf16(tmem + 0, td, sw128_desc(sb + kk * 2048, 16384, 1024), idesc_bf16(128, 128, 0, 1),
             kk > 0);
    mma_bf16(tmem + 128, sw128_desc(sb + Ly::kV + kk * 2048, 8192, 1024), td,
             idesc_bf16(128, 64, 1, 0), kk > 0);
  }
}

// W (rows 0..63 of tmem[0, 128)) as bf16 [token][channel] (K-major W, or the
// MN-major view with K = token).
__device__ __forceinline__ void extract_w(uint32_t lane_base, int quarter, int colhalf, int lane,
                                          uint32_t w) {
  if (quarter >= 2) return;
  const int r = quarter * 32 + lane;
  float v[64];
  tmem_ld64(lane_base + colhalf * 64, v);
#pragma unroll
  for (int q8 = 0; q8 < 8; ++q8)
    st_shared_v4(w + colhalf * 8192 + sw128_chunk(r, q8), pack_bf16x2(v[q8 * 8], v[q8 * 8 + 1]),
                 pack_bf16x2(v[q8 * 8 + 2], v[q8 * 8 + 3]), pack_bf16x2(v[q8 * 8 + 4], v[q8 * 8 + 5]),
                 pack_bf16x2(v[q8 * 8 + 6], v[q8 * 8 + 7]));
}

template <int DV>
__global__ void __launch_bounds__(kThreads, 1)
    chunked_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                   const __grid_constant__ CUtensorMap tm_o,
                   const __grid_constant__ CUtensorMap tm_snap,
                   const __grid_constant__ CUtensorMap tm_pool, const ChunkArgs a) {
  using Ly = Layout<DV>;
  constexpr int NH = DV / 2;  // state columns per thread
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, colhalf = warp >> 2;
  const uint32_t sbase = smem_u32(smem);

  int item = blockIdx.x;
  const int dvb = item % a.n_dvb;
  item /= a.n_dvb;
  const int h = item % a.H;
  const int rank = item / a.H;
  const SeqMeta m = a.meta[a.order[rank]];
  if (!m.ok) return;
  if (sbase & 1023) {  // the swizzled layouts need a 1024-byte aligned base
    if (tid == 0) raise_error(a.err, ERR_TIMEOUT);
    return;
  }
  const int H = a.H, dv = a.dv, dv0 = dvb * DV;

  uint8_t *misc = smem + Ly::kMisc;
  const uint32_t bar_tma0 = sbase + Ly::kMisc + Ly::kBars;
  const uint32_t bar_mma = bar_tma0 + 16;
  float *s_beta = reinterpret_cast<float *>(misc + Ly::kBeta);
  float *s_tot = reinterpret_cast<float *>(misc + Ly::kTot);
  float *s_anc = reinterpret_cast<float *>(misc + Ly::kAnc);
  float *s_gpart = reinterpret_cast<float *>(smem + Ly::kGpart);

  if (tid == 0) {
    mbar_init(bar_tma0, 1);
    mbar_init(bar_tma0 + 8, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_g);
    prefetch_tmap(&tm_o);
  }
  if (warp == 0) tmem_alloc(sbase + Ly::kMisc + Ly::kSlot, kTmemCols);
  // [T; M] starts at zero: the blocks of T above its diagonal are never written
  for (int e = tid; e < 16384 / 16; e += kThreads) st_shared_v4(sbase + Ly::kTM + 16 * e, 0, 0, 0, 0);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(misc + Ly::kSlot);
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
  // this thread's NH accumulator columns of a TMEM row, with a single wait
  auto ld_row = [](uint32_t taddr, float (&v)[NH]) {
    if constexpr (NH == 64) {
      tmem_ld64(taddr, v);
    } else {
      tmem_ld32(taddr, v);
    }
  };

  // ---- state rows owned by this thread: row c, columns [col0, col0 + NH)
  const int c = quarter * 32 + lane;
  const int col0 = colhalf * NH;
  float S[NH];
  {
    if (m.src >= 0) {
      const float4 *s0 = reinterpret_cast<const float4 *>(
          a.pool + (((int64_t)m.src * H + h) * kDK + c) * dv + dv0 + col0);
#pragma unroll
      for (int j = 0; j < NH / 4; ++j) {
        const float4 t = s0[j];
        S[4 * j] = t.x; S[4 * j + 1] = t.y; S[4 * j + 2] = t.z; S[4 * j + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < NH; ++j) S[j] = 0.f;
    }
  }

  const int nchunks = (m.len + kC - 1) / kC;
  const uint32_t tx_bytes = (6 + DV / 64) * 8192;
  auto issue_tma = [&](int n) {
    const int st = n & 1;
    const uint32_t sb = sbase + st * Ly::kStage;
    const uint32_t bar = bar_tma0 + 8 * st;
    const int y = m.tok0 + n * kC;
    mbar_expect_tx(bar, tx_bytes);
    tma_load_2d(sb + 0, &tm_k, h * kDK, y, bar);
    tma_load_2d(sb + 16384, &tm_k, h * kDK + 64, y, bar);
    tma_load_2d(sb + Ly::kQ, &tm_q, h * kDK, y, bar);
    tma_load_2d(sb + Ly::kQ + 16384, &tm_q, h * kDK + 64, y, bar);
#pragma unroll
    for (int j = 0; j < DV / 64; ++j)
      tma_load_2d(sb + Ly::kV + j * 8192, &tm_v, h * dv + dv0 + 64 * j, y, bar);
    tma_load_2d(sb + Ly::kG, &tm_g, h * kDK, y, bar);
    tma_load_2d(sb + Ly::kG + 8192, &tm_g, h * kDK + 64, y, bar);
  };

  bool tma_pending[2] = {false, false};
  uint32_t tma_parity[2] = {0, 0};  // parity the pending load of each stage completes with
  uint32_t mma_phase = 0;
  bool mma_pending = false;
  bool aborted = false;
  bool flagged = false;  // a chunk's decay left the exponent range: recomputed exactly later
  if (tid == 0 && nchunks > 0) issue_tma(0);
  tma_pending[0] = nchunks > 0;

  const uint32_t idesc_v = idesc_bf16(128, DV, 0, 1);
  const uint32_t idesc_vneg = idesc_bf16(128, DV, 0, 1, 1);
  const uint32_t idesc_ke = idesc_bf16(128, DV, 1, 1);

  // beta of row tid (threads 0..63) of the next kBetaAhead chunks, loaded
  // in one burst every kBetaAhead chunks (a register load in flight holds up
  // the next barrier, so its latency is paid once per burst)
  constexpr int kBetaAhead = 8;
  float beta_q[kBetaAhead];
  const int snap_every = a.snap_interval > 0 ? a.snap_interval / kC : 0;
  int snap_left = snap_every;
  int64_t snap_next = m.snap_off;
  int64_t snap_y = -1;  // row of a snapshot staged for a TMA store this chunk
#pragma unroll 1
  for (int n = 0; n < nchunks; ++n) {
    const int st = n & 1;
    uint8_t *stage = smem + st * Ly::kStage;
    const uint32_t sb = sbase + st * Ly::kStage;
    const int t0 = m.tok0 + n * kC;
    const int cl = min(kC, m.len - n * kC);
    if (n % kBetaAhead == 0) {
#pragma unroll
      for (int k = 0; k < kBetaAhead; ++k)
        beta_q[k] = (tid < 64 && n + k < nchunks)
                        ? load_beta(a.beta + (int64_t)(t0 + k * kC) * H + h, H,
                                    min(kC, m.len - (n + k) * kC), tid)
                        : 0.f;
    }
    const float beta_n = beta_q[0];
#pragma unroll
    for (int k = 0; k + 1 < kBetaAhead; ++k) beta_q[k] = beta_q[k + 1];

    if (!cta_wait(bar_tma0 + 8 * st, (n >> 1) & 1)) { aborted = true; break; }
    tma_pending[st] = false;

    // ------------------------------------------------------------ prep
    if (prep_chunk<Ly, DV>(sb, cl, beta_n, s_gpart, s_beta, s_tot, s_anc, tid) && !flagged) {
      flagged = true;
      if (tid == 0) atomicExch(a.rerun + rank * H + h, a.epoch);
    }

    // ------------------------------------------------------------ MMA1
    if (tid == 0) {
      issue_mma1<Ly>(tmem + 256, sb);
      mma_commit(bar_mma);
    }
    mma_pending = true;
    {  // S0' = Diag(e^{a}) S as the bf16 operand (MN-major: row = channel c), under MMA1
      const float ea = expf(s_anc[c]);
#pragma unroll
      for (int j = 0; j < NH / 8; ++j) {
        const int col = col0 + 8 * j;
        st_shared_v4(sbase + Ly::kS0 + (col >> 6) * 16384 + sw128_chunk(c, (col & 63) >> 3),
                     pack_bf16x2(ea * S[8 * j], ea * S[8 * j + 1]),
                     pack_bf16x2(ea * S[8 * j + 2], ea * S[8 * j + 3]),
                     pack_bf16x2(ea * S[8 * j + 4], ea * S[8 * j + 5]),
                     pack_bf16x2(ea * S[8 * j + 6], ea * S[8 * j + 7]));
      }
      fence_async_smem();
    }
    // the previous chunk's outputs were stored from the W buffer, which this
    // chunk's W overwrites after MMA2
    if (tid == 0) bulk_wait_read<0>();
    if (!cta_wait(bar_mma, mma_phase)) { aborted = true; break; }
    mma_phase ^= 1;
    mma_pending = false;
    tc_fence_after();

    // A (rows 0..63) into the solve's operands; M (rows 64..127) into [T; M]
    float *A10 = reinterpret_cast<float *>(smem + Ly::kU + 8192);
    extract_am(lane_base + 256, quarter, colhalf, lane, s_beta, A10,
               reinterpret_cast<float *>(smem + Ly::kLT), sbase + Ly::kTM);
    tc_fence_before();
    __syncthreads();

    // O = Q+ S0' runs on the tensor cores while the CUDA cores solve for T
    // (the commit after MMA2 covers it)
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tmem + 384,
                 sw128_desc(sb + Ly::kQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                 sw128_desc(sbase + Ly::kS0 + kk * 2048, 16384, 1024), idesc_v, kk > 0);
    }

    // ------------------------------------------------------------ solve
    // the next chunk's tiles go to the other stage (released at the end of
    // chunk n-1), requested by a thread that the solve leaves idle
    auto next_tiles = [&](int e) {
      if (e == 0 && n + 1 < nchunks) issue_tma(n + 1);
    };
    if (!solve_T(reinterpret_cast<const float *>(smem + Ly::kLT),
                 reinterpret_cast<float *>(smem + Ly::kU), A10,
                 reinterpret_cast<float *>(smem + Ly::kXd), reinterpret_cast<float *>(smem + Ly::kYt),
                 s_beta, smem + Ly::kTM, tmem, bar_mma, mma_phase, mma_pending, tid, next_tiles)) {
      aborted = true;
      break;
    }
    if (n + 1 < nchunks) {
      tma_pending[(n + 1) & 1] = true;
      tma_parity[(n + 1) & 1] = ((n + 1) >> 1) & 1;
    }

    // ------------------------------------------------------------ MMA2
    if (tid == 0) {
      issue_mma2<Ly, DV>(tmem, sbase + Ly::kTM, sb);
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!cta_wait(bar_mma, mma_phase)) { aborted = true; break; }
    mma_phase ^= 1;
    mma_pending = false;
    tc_fence_after();

    // W (rows 0..63) -> bf16 K-major operand
    extract_w(lane_base, quarter, colhalf, lane, sbase + Ly::kW);
    tc_fence_before();
    fence_async_smem();
    __syncthreads();

    // ------------------------------------------------------------ MMA3
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t bd = sw128_desc(sbase + Ly::kS0 + kk * 2048, 16384, 1024);
        mma_bf16(tmem + 128, sw128_desc(sbase + Ly::kW + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024),
                 bd, idesc_vneg, 1);
      }
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!cta_wait(bar_mma, mma_phase)) { aborted = true; break; }
    mma_phase ^= 1;
    mma_pending = false;
    tc_fence_after();

    // U (rows 0..63) -> bf16 MN-major operand (row = token)
    if (quarter < 2) {
      const int r = quarter * 32 + lane;
      float v[NH];
      ld_row(lane_base + 128 + col0, v);
#pragma unroll
      for (int q8 = 0; q8 < NH / 8; ++q8) {
        const int col = col0 + q8 * 8;
        st_shared_v4(sbase + Ly::kU + (col >> 6) * 8192 + sw128_chunk(r, (col & 63) >> 3),
                     pack_bf16x2(v[q8 * 8], v[q8 * 8 + 1]), pack_bf16x2(v[q8 * 8 + 2], v[q8 * 8 + 3]),
                     pack_bf16x2(v[q8 * 8 + 4], v[q8 * 8 + 5]),
                     pack_bf16x2(v[q8 * 8 + 6], v[q8 * 8 + 7]));
      }
    }
    tc_fence_before();
    fence_async_smem();
    __syncthreads();

    // ------------------------------------------------------------ MMA4
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bd = sw128_desc(sbase + Ly::kU + kk * 2048, 8192, 1024);
        mma_bf16(tmem + 256, sw128_desc(sb + Ly::kG + kk * 2048, 8192, 1024), bd, idesc_ke,
                 kk > 0);
        mma_bf16(tmem + 384, sw128_desc(sbase + Ly::kTM + 8192 + kk * 32, 16, 1024), bd, idesc_v,
                 1);
      }
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!cta_wait(bar_mma, mma_phase)) { aborted = true; break; }
    mma_phase ^= 1;
    mma_pending = false;
    tc_fence_after();

    // ------------------------------------------------------------ outputs
    // a whole chunk is staged in the W buffer (free since MMA3) as 128-byte
    // swizzled halves of 64 value columns and leaves with TMA stores after
    // the chunk's closing barrier; a ragged last chunk is written directly
    // (a full box would run into the next sequence's rows)
    if (quarter < 2) {
      const int r = quarter * 32 + lane;
      float v[NH];
      ld_row(lane_base + 384 + col0, v);
      if (cl == kC) {
#pragma unroll
        for (int q8 = 0; q8 < NH / 8; ++q8) {
          const int col = col0 + 8 * q8;
          st_shared_v4(sbase + Ly::kW + (col >> 6) * 8192 + sw128_chunk(r, (col & 63) >> 3),
                       pack_bf16x2(v[q8 * 8], v[q8 * 8 + 1]), pack_bf16x2(v[q8 * 8 + 2], v[q8 * 8 + 3]),
                       pack_bf16x2(v[q8 * 8 + 4], v[q8 * 8 + 5]),
                       pack_bf16x2(v[q8 * 8 + 6], v[q8 * 8 + 7]));
        }
        fence_async_smem();
      } else if (r < cl) {
        uint4 *dst = reinterpret_cast<uint4 *>(a.out + ((int64_t)(t0 + r) * H + h) * dv + dv0 + col0);
#pragma unroll
        for (int q8 = 0; q8 < NH / 8; ++q8)
          dst[q8] = make_uint4(pack_bf16x2(v[q8 * 8], v[q8 * 8 + 1]),
                               pack_bf16x2(v[q8 * 8 + 2], v[q8 * 8 + 3]),
                               pack_bf16x2(v[q8 * 8 + 4], v[q8 * 8 + 5]),
                               pack_bf16x2(v[q8 * 8 + 6], v[q8 * 8 + 7]));
      }
    }
    {
      // S = Diag(e^{G_C}) S + Diag(e^{G_C - a}) (K-^T U)   (K_end = K- e^{G_C - a})
      const float egc = expf(s_tot[c]), cke = expf(s_tot[c] - s_anc[c]);
      float v[NH];
      ld_row(lane_base + 256 + col0, v);
#pragma unroll
      for (int j = 0; j < NH; ++j) S[j] = fmaf(egc, S[j], cke * v[j]);
      // a snapshot after every snap_every full chunks (the interval is a
      // multiple of the chunk, so a ragged last chunk never ends on one)
      if (snap_every > 0 && --snap_left == 0 && cl == kC) {
        snap_left = snap_every;
        const int64_t s = snap_next++;
        if (s < a.snaps_capacity) {
          float *base = snapshot_base(a.snaps, a.snap_slots, a.pool, s, H, h, (int64_t)kDK * dv);
          if (base && a.snap_tma) {
            // staged in this chunk's input stage (dead since MMA4; its next
            // load waits for the store) as 128-byte swizzled boxes of 32
            // columns, then TMA-stored after the closing barrier
#pragma unroll
            for (int j = 0; j < NH / 4; ++j) {
              const int col = col0 + 4 * j;
              st_shared_v4(sb + (col >> 5) * 16384 + sw128_chunk(c, (col & 31) >> 2),
                           __float_as_uint(S[4 * j]), __float_as_uint(S[4 * j + 1]),
                           __float_as_uint(S[4 * j + 2]), __float_as_uint(S[4 * j + 3]));
            }
            fence_async_smem();
            snap_y = a.snap_slots ? ((int64_t)a.snap_slots[s] * H + h) * kDK : (s * H + h) * kDK;
          } else if (base) {
            float4 *dst = reinterpret_cast<float4 *>(base + (int64_t)c * dv + dv0 + col0);
#pragma unroll
            for (int j = 0; j < NH / 4; ++j)
              dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
          }
        } else if (tid == 0) {
          raise_error(a.err, ERR_SNAP_CAPACITY);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && cl == kC) {
#pragma unroll
      for (int j = 0; j < DV / 64; ++j)
        tma_store_2d(&tm_o, sbase + Ly::kW + j * 8192, h * dv + dv0 + 64 * j, t0);
      if (snap_y >= 0) {
#pragma unroll
        for (int j = 0; j < DV / 32; ++j)
          tma_store_2d(a.snap_slots ? &tm_pool : &tm_snap, sb + j * 16384, dv0 + 32 * j,
                       (int)snap_y);
      }
      bulk_commit();
    }
    snap_y = -1;
  }

  if (tid == 0) bulk_wait<0>();  // every output store complete (and its source read)
  if (aborted) {
    if (tid == 0) raise_error(a.err, ERR_TIMEOUT);
    // drain what is still in flight (bounded), then release TMEM
    for (int s = 0; s < 2; ++s)
      if (tma_pending[s]) mbar_wait(bar_tma0 + 8 * s, tma_parity[s]);
    if (mma_pending) mbar_wait(bar_mma, mma_phase);
  } else if (!flagged) {  // a flagged unit keeps its source for the exact recomputation
    float4 *dst = reinterpret_cast<float4 *>(
        a.pool + (((int64_t)m.dst * H + h) * kDK + c) * dv + dv0 + col0);
#pragma unroll
    for (int j = 0; j < NH / 4; ++j)
      dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ cooperative mode
// For batches with few (sequence, head) pairs, one CTA per pair carries that
// pair's state ("chain" CTA) while every other CTA of a cooperative grid
// prepares chunks ("producer" CTAs): the part of a chunk that does not depend
// on its start state.  Producers take chunks in ticket order (chunk index
// major, so all pairs advance together) and hand each to its pair's chain CTA
// as a package in a ring of kCoopRing slots in global memory (small enough to
// stay in L2).  Ready / consumed flags hold the call's epoch in their upper
// 32 bits and the chunk number + 1 below; every wait is bounded and an abort
// word stops all CTAs after a timeout.
//
// The single-CTA kernel's update is, with S' = Diag(e^{a}) S,
//     U = U~ - W S',  S_next = Diag(e^{G_C}) S + Diag(e^{G_C - a}) K-^T U,
//     O = Q+ S' + M U.
// The producer folds the per-channel factors into its operands,
//     K^  = K- Diag(e^{G_C - a})   (= K Diag(e^{G_C - G_r}) per row: at most |K|)
//     W^  = W Diag(e^{a}),  Q+' = Q+ Diag(e^{a}),
// so that with the state itself as the bf16 operand
//     U = U~ - W^ S,   S_next = Diag(e^{G_C}) S + K^^T U,   O = Q+' S + M U,
// and the chain CTA works on the transposed state: S^T (bf16, in TMEM) is the
// A operand of [X^T | O^T] = S^T [W^; Q+']^T (one product of N = 128: a
// tensor-core instruction with N <= 128 costs about 94 cycles whatever its M
// and N, measured on GB300, so two products of N = 64 cost twice as much);
// the state warps form
// U^T = U~^T - X^T (bf16, in TMEM), the A operand of acc^T = U^T K^ and of
// O^T += U^T M^T.

// package layout (bytes); each operand in the shared-memory layout the chain
// CTA feeds to its MMAs (U~ is read by its state warps), copied verbatim
// per channel half h: W^ [64 tok][64 ch] at 16384 h and Q+' [64 tok][64 ch] at
// 16384 h + 8192 (bf16, K-major), i.e. the 128 rows of one B operand [W^; Q+']
constexpr uint32_t kPkWQ = 0;
constexpr uint32_t kPkKm = 32768;   // K^ [64 tok][128 ch] bf16, 2 halves x 8 KiB
constexpr uint32_t kPkU = 49152;    // U~^T [128 dv][64 tok] bf16, 128-byte swizzled rows
constexpr uint32_t kPkM = 65536;    // M [64 tok][64 tok] bf16, K-major, 8 KiB
constexpr uint32_t kPkDec = 73728;  // f32 e^{G_C}[128]
static_assert(kPkDec + 512 <= kCoopPkgBytes && kCoopPkgBytes % 1024 == 0, "package layout");
// a package is fetched as kPkPieces bulk copies of kPkPiece bytes (8 measured
// 0.3-0.6% faster than 4, measured back to back on one GPU)
constexpr uint32_t kPkPieces = 8, kPkPiece = (uint32_t)kCoopPkgBytes / kPkPieces;
static_assert(kPkPiece % 16 == 0 && kPkPiece * kPkPieces == kCoopPkgBytes, "bulk copy pieces");
// chain CTA shared memory: three package stages (a package copy from L2
// takes about as long as a chunk's state step, so two stages leave the chain
// waiting for its next package), mbarriers, TMEM slot
constexpr int kChStages = 3;
constexpr uint32_t kChMisc = kChStages * (uint32_t)kCoopPkgBytes;
constexpr uint32_t kChBytes = kChMisc + 192;
constexpr uint32_t kCoopSmem =
    Layout<128>::kBytes > kChBytes ? Layout<128>::kBytes : kChBytes;

struct CoopArgs {
  ChunkArgs c;
  uint8_t *ring;                       // [units][kCoopRing][kCoopPkgBytes]
  unsigned long long *ready;           // [units][kCoopRing]
  unsigned long long *consumed;        // [split][units][kCoopRing], one per chain CTA
  uint32_t *hdr;                       // [0] ticket, [1] abort, [2] max chunks per sequence
  int units;                           // (sequence, head) pairs
  int split;                           // chain CTAs per pair: 1 (whole state) or 2 (column halves)
  uint32_t epoch;
};

__device__ __forceinline__ unsigned long long coop_tag(uint32_t epoch, int n) {
  return ((unsigned long long)epoch << 32) | (unsigned long long)(n + 1);
}

// Thread 0: bounded wait until *p >= want (about a second); false on timeout
// or when another CTA aborted.
__device__ bool coop_flag_wait(const unsigned long long *p, unsigned long long want,
                               const uint32_t *abort_flag) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    if (ld_acquire_u64(p) >= want) return true;
    if (*reinterpret_cast<const volatile uint32_t *>(abort_flag)) return false;
    __nanosleep(i < 64 ? 32 : 256);
  }
  return false;
}

__device__ __forceinline__ void coop_abort(const CoopArgs &a) {
  atomicExch(a.hdr + 1, 1u);
  raise_error(a.c.err, ERR_TIMEOUT);
}

__device__ __forceinline__ uint4 pack8(const float *v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}


// Producer role: prepares chunks of any pair, in ticket order.
__device__ void coop_producer(uint8_t *smem, const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                              const CUtensorMap *tm_v, const CUtensorMap *tm_g,
                              const CoopArgs &a) {
  using Ly = Layout<128>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, colhalf = warp >> 2;
  const uint32_t sbase = smem_u32(smem);
  const int H = a.c.H, units = a.units;
  uint8_t *misc = smem + Ly::kMisc;
  const uint32_t bar_tma0 = sbase + Ly::kMisc + Ly::kBars, bar_mma = bar_tma0 + 16;
  float *s_beta = reinterpret_cast<float *>(misc + Ly::kBeta);
  float *s_tot = reinterpret_cast<float *>(misc + Ly::kTot);
  float *s_anc = reinterpret_cast<float *>(misc + Ly::kAnc);
  float *s_ea = reinterpret_cast<float *>(misc + Ly::kEa);
  // e^{G_C - a}: in the solve scratch, which is free while the first MMA runs
  float *s_cka = reinterpret_cast<float *>(smem + Ly::kScr);
  float *s_cke = reinterpret_cast<float *>(misc + Ly::kCke);
  float *s_gpart = reinterpret_cast<float *>(smem + Ly::kGpart);
  int2 *s_seq = reinterpret_cast<int2 *>(misc + Ly::kSeqs);  // (tok0, len or 0) per sequence
  volatile int *s_item = reinterpret_cast<volatile int *>(misc + 32);

  for (int r = tid; r < units / H; r += kThreads) {
    const SeqMeta m = a.c.meta[a.c.order[r]];
    s_seq[r] = make_int2(m.tok0, m.ok ? m.len : 0);
  }
  if (tid == 0) {
    prefetch_tmap(tm_q);
    prefetch_tmap(tm_k);
    prefetch_tmap(tm_v);
    prefetch_tmap(tm_g);
  }
  if (tid == 0) {
    mbar_init(bar_tma0, 1);
    mbar_init(bar_tma0 + 8, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(sbase + Ly::kMisc + Ly::kSlot, kTmemCols);
  for (int e = tid; e < 16384 / 16; e += kThreads) st_shared_v4(sbase + Ly::kTM + 16 * e, 0, 0, 0, 0);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(misc + Ly::kSlot);
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
  const int total = (int)a.hdr[2] * units;

  // Tickets come from a global counter (chunk index major).  A producer
  // works through its tickets in increasing order and a ticket only ever
  // waits for smaller ones, so the smallest unfinished ticket can always
  // proceed.  take_from(t) validates a raw ticket, drawing again past
  // chunks beyond a sequence's end.
  auto valid = [&](int t) { return (t / units) * kC < s_seq[(t % units) / H].y; };
  auto take_from = [&](int t) -> int {  // thread 0
    while (t < total && !valid(t)) t = (int)atomicAdd(a.hdr, 1u);
    return t < total ? t : -1;
  };
  auto take = [&]() -> int { return take_from((int)atomicAdd(a.hdr, 1u)); };
  // TMA loads of chunk t into stage st, one thread: the k, v and g tiles
  // (with the byte count of all eight) and the q tiles, which the producer
  // may request at different points
  auto issue_kvg = [&](int t, int st) {
    const int u = t % units, h = u % H;
    const uint32_t sb = sbase + st * Ly::kStage, bar = bar_tma0 + 8 * st;
    const int y = s_seq[u / H].x + (t / units) * kC;
    mbar_expect_tx(bar, 8 * 8192);
    tma_load_2d(sb, tm_k, h * kDK, y, bar);
    tma_load_2d(sb + 16384, tm_k, h * kDK + 64, y, bar);
    tma_load_2d(sb + Ly::kV, tm_v, h * 128, y, bar);
    tma_load_2d(sb + Ly::kV + 8192, tm_v, h * 128 + 64, y, bar);
    tma_load_2d(sb + Ly::kG, tm_g, h * kDK, y, bar);
    tma_load_2d(sb + Ly::kG + 8192, tm_g, h * kDK + 64, y, bar);
  };
  auto issue_q = [&](int t, int st) {
    const int u = t % units, h = u % H;
    const uint32_t sb = sbase + st * Ly::kStage, bar = bar_tma0 + 8 * st;
    const int y = s_seq[u / H].x + (t / units) * kC;
    tma_load_2d(sb + Ly::kQ, tm_q, h * kDK, y, bar);
    tma_load_2d(sb + Ly::kQ + 16384, tm_q, h * kDK + 64, y, bar);
  };
  auto issue = [&](int t, int st) {
    issue_kvg(t, st);
    issue_q(t, st);
  };

  // the tiles of a chunk are loaded while the chunk before it is worked on:
  // each chunk's tiles are requested at the end of the chunk two before it,
  // into the stage that chunk used (the first two up front)
  if (tid == 0) {
    const int t0 = take();
    s_item[0] = t0;
    s_item[1] = t0 >= 0 ? take() : -1;
    if (t0 >= 0) issue(t0, 0);
    if (s_item[1] >= 0) issue(s_item[1], 1);
  }
  __syncthreads();
  int cur = s_item[0], next = s_item[1];
  // beta of chunk t, row tid (threads 0..63); a chunk's beta is loaded at the
  // end of the chunk before it, where its latency hides under thread 0's
  // slot wait and copy issue that the closing barrier waits for anyway
  auto beta_of = [&](int t) -> float {
    if (tid >= 64 || t < 0) return 0.f;
    const int tn = t / units, tu = t % units;
    const int2 tq = s_seq[tu / H];
    return load_beta(a.c.beta + (int64_t)(tq.x + tn * kC) * H + tu % H, H,
                     min(kC, tq.y - tn * kC), tid);
  };
  float beta_r = beta_of(cur);
  uint32_t uses[2] = {0, 0}, mma_phase = 0;
  bool tma_pending[2] = {cur >= 0, next >= 0}, mma_pending = false, aborted = false;
  // Thread kLoad requests the tiles of the chunk two ahead at the end of a
  // chunk; thread kPub then waits for the ring slot and stores the package
  // with bulk copies (shared -> global bulk writes run at about 29 B/cycle per
  // SM, so the loads go first).  At the next chunk's first MMA kPub waits
  // until the stores are complete (their sources are then free) and publishes
  // the package (ready flag): its proxy fence then has no tile loads of its
  // own in flight to order.  Thread 0 issues the MMAs and takes tickets.
  constexpr int kPub = 64, kLoad = 96;
  bool pend = false;
  unsigned long long *pend_flag = nullptr, pend_tag = 0, slot_seen = 0;
  int raw_ticket = 0;  // thread 0: drawn at a chunk's first MMA, validated at its second
  for (int it = 0; cur >= 0; ++it) {
    const int st = it & 1;
    const int n = cur / units, u = cur % units;
    const int cl = min(kC, s_seq[u / H].y - n * kC);
    const uint32_t sb = sbase + st * Ly::kStage;
    const float beta_n = beta_r;
    if (!cta_wait(bar_tma0 + 8 * st, uses[st] & 1)) { aborted = true; break; }
    ++uses[st];
    tma_pending[st] = false;

    if (prep_chunk<Ly, 128>(sb, cl, beta_n, s_gpart, s_beta, s_tot, s_anc, tid) && tid == 0) {
      // the flag is written before this chunk's package is published, so the
      // pair's chain CTA sees it by the time it has taken its last package
      atomicExch(a.c.rerun + u, a.epoch);
      __threadfence();
    }
    if (tid == 0) {
      issue_mma1<Ly>(tmem + 256, sb);
      mma_commit(bar_mma);
      raw_ticket = next >= 0 ? (int)atomicAdd(a.hdr, 1u) : total;  // used at MMA2
    }
    if (tid < 128) {
      s_ea[tid] = expf(s_anc[tid]);
      s_cka[tid] = expf(s_tot[tid] - s_anc[tid]);
    }
    // While the first MMA runs, every warp but thread kPub's stages K^ = K-
    // Diag(e^{G_C - a}), which needs only the prepared tiles, into the upper
    // half of the S0 region.  That warp lets the others start (named barrier
    // 1) once the previous package's bulk stores have read their sources,
    // then waits until those stores are complete and publishes the package.
    constexpr int kStagers = kThreads - 32;
    if (warp == kPub / 32) {
      if (tid == kPub) bulk_wait_read<0>();
      __syncwarp();
      named_bar_arrive(1, kThreads);
      if (tid == kPub) {
        bulk_wait<0>();
        if (pend) {
          fence_proxy_async_all();
          st_release_u64(pend_flag, pend_tag);
          pend = false;
        }
      }
    } else {
      named_bar_sync(1, kThreads);
      for (int e = tid - (warp > kPub / 32 ? 32 : 0); e < 1024; e += kStagers) {
        const int half = e >> 9, r = (e >> 3) & 63, q = e & 7;
        const uint32_t off = r * 128 + q * 16;
        const float4 *f = reinterpret_cast<const float4 *>(s_cka + half * 64 + 8 * (q ^ (r & 7)));
        const float4 f0 = f[0], f1 = f[1];
        const uint4 w = ld_shared_v4(sb + Ly::kG + half * 8192 + off);
        st_shared_v4(sbase + Ly::kS0 + 16384 + half * 8192 + off,
                     pack_bf16x2(bf16lo(w.x) * f0.x, bf16hi(w.x) * f0.y),
                     pack_bf16x2(bf16lo(w.y) * f0.z, bf16hi(w.y) * f0.w),
                     pack_bf16x2(bf16lo(w.z) * f1.x, bf16hi(w.z) * f1.y),
                     pack_bf16x2(bf16lo(w.w) * f1.z, bf16hi(w.w) * f1.w));
      }
    }
    mma_pending = true;
    if (!cta_wait(bar_mma, mma_phase)) { aborted = true; break; }
    mma_phase ^= 1;
    mma_pending = false;
    tc_fence_after();
    float *A10 = reinterpret_cast<float *>(smem + Ly::kU + 8192);
    extract_am(lane_base + 256, quarter, colhalf, lane, s_beta, A10,
               reinterpret_cast<float *>(smem + Ly::kLT), sbase + Ly::kTM);
    tc_fence_before();
    __syncthreads();
    if (!solve_T(reinterpret_cast<const float *>(smem + Ly::kLT),
                 reinterpret_cast<float *>(smem + Ly::kU), A10,
                 reinterpret_cast<float *>(smem + Ly::kXd), reinterpret_cast<float *>(smem + Ly::kYt),
                 s_beta, smem + Ly::kTM, tmem, bar_mma, mma_phase, mma_pending, tid, [](int) {})) {
      aborted = true;
      break;
    }
    if (tid == 0) {
      issue_mma2_coop<Ly>(tmem, sbase + Ly::kTM, sb);
      mma_commit(bar_mma);
    }
    // while the second MMA runs, Q+' = Q+ Diag(e^{a}) into the lower half of
    // the S0 region
    for (int e = tid; e < 1024; e += kThreads) {
      const int half = e >> 9, r = (e >> 3) & 63, q = e & 7;
      const uint32_t off = r * 128 + q * 16;
      const float4 *f = reinterpret_cast<const float4 *>(s_ea + half * 64 + 8 * (q ^ (r & 7)));
      const float4 f0 = f[0], f1 = f[1];
      const uint4 w = ld_shared_v4(sb + Ly::kQ + half * 16384 + off);
      st_shared_v4(sbase + Ly::kS0 + half * 8192 + off,
                   pack_bf16x2(bf16lo(w.x) * f0.x, bf16hi(w.x) * f0.y),
                   pack_bf16x2(bf16lo(w.y) * f0.z, bf16hi(w.y) * f0.w),
                   pack_bf16x2(bf16lo(w.z) * f1.x, bf16hi(w.z) * f1.y),
                   pack_bf16x2(bf16lo(w.w) * f1.z, bf16hi(w.w) * f1.w));
    }
    if (tid == 0) s_item[2] = next >= 0 ? take_from(raw_ticket) : -1;
    if (tid == kPub && n >= kCoopRing) {  // peek at this chunk's ring slot early; it is waited
      // for only if a chain CTA of the pair had not yet copied out the chunk that used it before
      slot_seen = ld_relaxed_u64(a.consumed + u * kCoopRing + n % kCoopRing);
      for (int hv = 1; hv < a.split; ++hv)
        slot_seen = min(slot_seen,
                        ld_relaxed_u64(a.consumed + ((size_t)hv * units + u) * kCoopRing + n % kCoopRing));
    }
    mma_pending = true;
    if (!cta_wait(bar_mma, mma_phase)) { aborted = true; break; }
    mma_phase ^= 1;
    mma_pending = false;
    const int after = s_item[2];
    tc_fence_after();
    // The package is staged in shared memory in its final layout, outside
    // both input stages, then written out with bulk copies: W^ = W Diag(e^{a})
    // in the W buffer, U~^T in the U buffer, K^ and Q+' in the S0 region (staged
    // beside the first and the second MMA), M where the solve left it and
    // e^{G_C} in its own vector.
    // the chunk two ahead goes to this chunk's stage: its k, v and g tiles are
    // dead now (its q tiles are requested last, just before the package
    // stores), and thread kPub's warp has no rows to stage
    if (tid == kLoad && after >= 0) issue_kvg(after, st);
    if (after >= 0) tma_pending[st] = true;
    {  // U~^T: TMEM lane = value column c, this warp's 32 tokens -> row c of kU
      const int c = quarter * 32 + lane;
      float v[32];
      tmem_ld32(lane_base + 128 + colhalf * 32, v);
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        const uint4 w = pack8(v + 8 * q8);
        st_shared_v4(sbase + Ly::kU + sw128_chunk(c, colhalf * 4 + q8), w.x, w.y, w.z, w.w);
      }
    }
    if (quarter < 2) {  // W^: rows 0..63 of tmem[0, 128)
      const int r = quarter * 32 + lane;
      float v[64];
      tmem_ld64(lane_base + colhalf * 64, v);
      const float4 *ea = reinterpret_cast<const float4 *>(s_ea + colhalf * 64);
#pragma unroll
      for (int q4 = 0; q4 < 16; ++q4) {
        const float4 e4 = ea[q4];
        v[4 * q4] *= e4.x;
        v[4 * q4 + 1] *= e4.y;
        v[4 * q4 + 2] *= e4.z;
        v[4 * q4 + 3] *= e4.w;
      }
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const uint4 w = pack8(v + 8 * q8);
        st_shared_v4(sbase + Ly::kW + colhalf * 8192 + sw128_chunk(r, q8), w.x, w.y, w.z, w.w);
      }
    }
    if (tid < 128) s_cke[tid] = expf(s_tot[tid]);  // e^{G_C} for the package
    tc_fence_before();
    fence_async_smem();  // the staged package, for the bulk stores
    const int slot = n % kCoopRing;
    {
      int ok = 1;
      __syncthreads();
      beta_r = beta_of(next);
      if (tid == kLoad && after >= 0) issue_q(after, st);  // before the stores
      if (tid == kPub && n >= kCoopRing && slot_seen < coop_tag(a.epoch, n - kCoopRing))
        for (int hv = 0; hv < a.split && ok; ++hv)
          ok = coop_flag_wait(a.consumed + ((size_t)hv * units + u) * kCoopRing + slot,
                              coop_tag(a.epoch, n - kCoopRing), a.hdr + 1);
      // the package, piece by piece from where it was staged (W, S0 region,
      // U, M, e^{G_C}); these are first overwritten after
      // the next chunk's first MMA, where thread kPub waits for the stores
      if (tid == kPub && ok) {
        uint8_t *pk = a.ring + ((size_t)u * kCoopRing + slot) * kCoopPkgBytes;
        bulk_s2g(pk + kPkWQ, sbase + Ly::kW, 8192);
        bulk_s2g(pk + kPkWQ + 8192, sbase + Ly::kS0, 8192);
        bulk_s2g(pk + kPkWQ + 16384, sbase + Ly::kW + 8192, 8192);
        bulk_s2g(pk + kPkWQ + 24576, sbase + Ly::kS0 + 8192, 8192);
        bulk_s2g(pk + kPkKm, sbase + Ly::kS0 + 16384, 16384);
        bulk_s2g(pk + kPkU, sbase + Ly::kU, 16384);
        bulk_s2g(pk + kPkM, sbase + Ly::kTM + 8192, 8192);
        bulk_s2g(pk + kPkDec, sbase + Ly::kMisc + Ly::kCke, 512);
        bulk_commit();
        pend = true;
        pend_flag = a.ready + u * kCoopRing + slot;
        pend_tag = coop_tag(a.epoch, n);
      }
      if (after >= 0) tma_pending[st] = true;
      if (__syncthreads_or(!ok)) { aborted = true; break; }
    }
    cur = next;
    next = after;
  }
  if (tid == kPub) {  // the last package: complete, then published (unless aborted)
    bulk_wait<0>();
    if (pend && !aborted) {
      fence_proxy_async_all();
      st_release_u64(pend_flag, pend_tag);
    }
  }
  if (aborted) {
    if (tid == 0) coop_abort(a);
    for (int s = 0; s < 2; ++s)
      if (tma_pending[s]) mbar_wait(bar_tma0 + 8 * s, uses[s] & 1);
    if (mma_pending) mbar_wait(bar_mma, mma_phase);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Chain role: carries the state of pair u through its packages, with its warps
// specialised:
//   warps 0-3 (state): thread j holds column j of S (row j of S^T) for all 128
//     channels in fp32 registers.  Per chunk n it stores bf16(S^T) into TMEM
//     (the A operand of the chunk's state-dependent product; the previous
//     chunk's, which read it, completed before that chunk's acc^T),
//     retires chunk n-1's outputs in two halves while X^T and acc^T run, forms
//     U^T = U~^T - X^T (bf16, into TMEM), then applies
//     S <- Diag(e^{G_C}) S + acc and writes snapshots.
//   warp 4, one lane (MMA): per chunk, once package n has landed it hands its
//     ring slot back to the producers; once S^T is stored, [X^T | O^T] =
//     S^T [W^; Q+']^T into buffer n & 1 (commit: X ready); once the state
//     warps stored U^T = U~^T - X^T, acc^T = U^T K^ (commit: acc ready) and
//     O^T += U^T M^T (commit: outputs ready, stage free).
//   warps 5-7, one lane each (loaders): warp 5 + k waits until package n =
//     k (mod 3) is in the ring and stage k is free, and requests it with bulk
//     copies; its next package's ready flag is read (acquire) while this one
//     is in flight.
// TMEM columns: acc^T [0, 128); [X^T | O^T][b] [128 + 128 b, +128); S^T as
// bf16 pairs [384, 448); U^T as bf16 pairs [448, 480).
// Every wait is bounded; a role that gives up raises the abort word and
// leaves its loop, and the others then time out.
// Warp-uniform bounded wait: every lane polls, and all lanes give up together
// if any did, so the warp stays converged for the tcgen05 loads and stores.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// State warps of a half chain: value columns [64 hv, 64 hv + 64) of pair u.
// The chain's MMAs then have M = 64, whose rows m sit in TMEM lane
// 32 (m / 16) + m % 16: warp w owns rows 16 w .. 16 w + 15 in the first 16
// lanes of its quarter and reaches them with the 16-lane shapes, so every
// thread works.  Thread t (g = t / 4, q = t % 4) holds value columns
// j0 = 64 hv + 16 w + g and j0 + 8 and, of each, channels 8 r + 2 q + {0, 1},
// r = 0..15: 64 state elements, half of a whole-column thread's 128.  The
// 16x256b loads of X^T and acc^T hand it exactly the tokens or channels that
// its 16x128b stores of U^T and S^T pack into one bf16 pair (column 4 r + q
// holds K-positions 8 r + 2 q, 8 r + 2 q + 1), so no value changes thread.
// Returns false when a wait gave up.
__device__ bool chain_state_half(uint8_t *smem, const CoopArgs &a, const CUtensorMap *tm_o, int u,
                                 int hv, const SeqMeta &m, int N, uint32_t tmem, uint32_t bars) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const uint32_t sbase = smem_u32(smem);
  const int H = a.c.H, h = u % H, dv = a.c.dv;
  const uint32_t full0 = bars, empty0 = bars + 24, sready0 = bars + 48, accf = bars + 64,
                 xf = bars + 72, of0 = bars + 80, oe0 = bars + 96, uready = bars + 120,
                 sreadyhi0 = bars + 136;
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  const int j0 = 64 * hv + 16 * warp + g;
  float S[2][32];  // S[s][2 r + e]: channel 8 r + 2 q + e of value column j0 + 8 s
  if (m.ok && m.src >= 0) {
    const float *s0 = a.c.pool + ((int64_t)m.src * H + h) * kDK * dv + j0;
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int i = 0; i < 32; ++i) S[s][i] = s0[(int64_t)(8 * (i >> 1) + 2 * q + (i & 1)) * dv + 8 * s];
  } else {
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int i = 0; i < 32; ++i) S[s][i] = 0.f;
  }
  // outputs of chunk n, half hf (tokens 32 hf .. 32 hf + 31), from O^T buffer
  // n & 1 with the 16x64b shape: register r is token 2 r + oc of value column
  // 64 hv + 16 w + orow.  A full half leaves through a TMA store per warp: its
  // 16 columns x 32 tokens as bf16 rows of 32 bytes (conflict-free 2-byte
  // shared stores, two tokens per instruction) in 1 KiB of package stage n % 3
  // that the loaders leave alone (the other column half's rows of U~^T), where
  // chunk n + 3 writes next once lane 0 saw the stores read it.  A ragged half
  // is stored element by element (rows past the sequence end belong to the
  // next sequence).
  const int orow = g + 8 * (lane & 1), oc = (lane >> 1) & 1;
  const uint32_t obuf = kPkU + 8192u * (1 - hv) + 2048u * warp;
  auto retire = [&](int n, int hf) -> bool {
    const int b = n & 1;
    if (hf == 0 && !warp_wait(of0 + 8 * b, (n >> 1) & 1)) return false;
    tc_fence_after();
    uint32_t v[16];
    tmem_ld16x64_x16(lane_base + 192 + 128 * b + 32 * hf, v);
    tmem_wait_ld();
    reg_fence16(v);
    if (hf == 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(oe0 + 8 * b);
    }
    const int cl = min(kC, m.len - n * kC) - 32 * hf;
    if (cl >= 32) {
      const uint32_t buf = (uint32_t)(n % kChStages) * (uint32_t)kCoopPkgBytes + obuf + 1024u * hf;
      if (hf == 0) {  // chunk n - 3's two stores (four groups since) have read both halves
        if (lane == 0) bulk_wait_read<4>();
        __syncwarp();
      }
#pragma unroll
      for (int r = 0; r < 16; ++r)
        *reinterpret_cast<__nv_bfloat16 *>(smem + buf + (2 * r + oc) * 32 + 2 * orow) =
            __float2bfloat16_rn(__uint_as_float(v[r]));
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tm_o, sbase + buf, h * dv + 64 * hv + 16 * warp, m.tok0 + n * kC + 32 * hf);
        bulk_commit();
      }
    } else {
      const int64_t ts = (int64_t)H * dv;
      __nv_bfloat16 *o = a.c.out + ((int64_t)(m.tok0 + n * kC + 32 * hf + oc) * H + h) * dv +
                         64 * hv + 16 * warp + orow;
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (2 * r + oc < cl) o[2 * r * ts] = __float2bfloat16_rn(__uint_as_float(v[r]));
    }
    return true;
  };
  auto store_state = [&](float *base) {  // a whole state's [dk][dv] fp32 layout
    float *d = base + j0;
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int i = 0; i < 32; ++i) d[(int64_t)(8 * (i >> 1) + 2 * q + (i & 1)) * dv + 8 * s] = S[s][i];
  };
  // bf16(S^T) channels [64 p, 64 p + 64) -> TMEM, then the half-p barrier of
  // chunk parity buf: the first product's first four MMAs (K = channels
  // 0..63) start while the second half of the state is still being updated
  auto store_st = [&](int buf, int p) {
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r[2 * i] = pack_bf16x2(S[0][16 * p + 2 * i], S[0][16 * p + 2 * i + 1]);
      r[2 * i + 1] = pack_bf16x2(S[1][16 * p + 2 * i], S[1][16 * p + 2 * i + 1]);
    }
    tmem_st16x128_x8(lane_base + 384 + 32 * p, r);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive((p ? sreadyhi0 : sready0) + 8 * buf);
  };
  const int snap_every = a.c.snap_interval > 0 ? a.c.snap_interval / kC : 0;
  int snap_left = snap_every;
  int64_t snap_next = m.snap_off;
  if (N > 0) {
    store_st(0, 0);
    store_st(0, 1);
  }
  for (int n = 0; n < N; ++n) {
    const int b = n & 1, st = n % kChStages;
    if (n > 0 && !retire(n - 1, 0)) return false;
    if (!warp_wait(full0 + 8 * st, (n / kChStages) & 1) || !warp_wait(xf, n & 1)) return false;
    tc_fence_after();
    const uint32_t sp = sbase + st * (uint32_t)kCoopPkgBytes;
    {  // U^T = U~^T - X^T: tokens 8 r + 2 q + {0, 1} of value columns j0, j0 + 8
      uint32_t x[32], w0[8], w1[8];
      tmem_ld16x256_x8(lane_base + 128 + 128 * b, x);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        w0[r] = ld_shared_u32(sp + kPkU + sw128_chunk(j0, r) + 4 * q);
        w1[r] = ld_shared_u32(sp + kPkU + sw128_chunk(j0 + 8, r) + 4 * q);
      }
      tmem_wait_ld();
      reg_fence(x);
      uint32_t ur[16];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        ur[2 * r] = pack_bf16x2(bf16lo(w0[r]) - __uint_as_float(x[4 * r]),
                                bf16hi(w0[r]) - __uint_as_float(x[4 * r + 1]));
        ur[2 * r + 1] = pack_bf16x2(bf16lo(w1[r]) - __uint_as_float(x[4 * r + 2]),
                                    bf16hi(w1[r]) - __uint_as_float(x[4 * r + 3]));
      }
      tmem_st16x128_x8(lane_base + 448, ur);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(uready);
    if (n > 0) retire(n - 1, 1);
    if (!warp_wait(accf, n & 1)) return false;
    tc_fence_after();
    {  // S = Diag(e^{G_C}) S + acc: channels 8 r + 2 q + {0, 1}, then S^T of the
       // next chunk into the other buffer (last read by chunk n - 1's MMAs, done
       // before X^T of chunk n completed), one channel half at a time
      const uint32_t egc = sp + kPkDec + 8 * q;
      uint32_t v[2][32];
      tmem_ld16x256_x8(lane_base, v[0]);
      tmem_ld16x256_x8(lane_base + 64, v[1]);
      tmem_wait_ld();
      reg_fence(v[0]);
      reg_fence(v[1]);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const int r = 8 * p + rr;
          const float2 e = ld_shared_f2(egc + 32 * r);
          S[0][2 * r] = fmaf(e.x, S[0][2 * r], __uint_as_float(v[p][4 * rr]));
          S[0][2 * r + 1] = fmaf(e.y, S[0][2 * r + 1], __uint_as_float(v[p][4 * rr + 1]));
          S[1][2 * r] = fmaf(e.x, S[1][2 * r], __uint_as_float(v[p][4 * rr + 2]));
          S[1][2 * r + 1] = fmaf(e.y, S[1][2 * r + 1], __uint_as_float(v[p][4 * rr + 3]));
        }
        if (n + 1 < N) store_st(b ^ 1, p);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    const int cl = min(kC, m.len - n * kC);
    if (snap_every > 0 && --snap_left == 0 && cl == kC) {
      snap_left = snap_every;
      const int64_t s = snap_next++;
      if (s < a.c.snaps_capacity) {
        float *base = snapshot_base(a.c.snaps, a.c.snap_slots, a.c.pool, s, H, h, (int64_t)kDK * dv);
        if (base) store_state(base);
      } else if (tid == 0 && hv == 0) {
        raise_error(a.c.err, ERR_SNAP_CAPACITY);
      }
    }
  }
  if (N > 0 && !(retire(N - 1, 0) && retire(N - 1, 1))) return false;
  // a unit flagged by a producer keeps its source for the exact recomputation
  const bool flagged = atomicAdd(a.c.rerun + u, 0u) == a.epoch;
  if (m.ok && !flagged) store_state(a.c.pool + ((int64_t)m.dst * H + h) * kDK * dv);
  return true;
}

template <bool kHalf>
__device__ void coop_chain(uint8_t *smem, const CoopArgs &a, const CUtensorMap *tm_o, int u, int hv) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  const int H = a.c.H, h = u % H, dv = a.c.dv;
  const SeqMeta m = a.c.meta[a.c.order[u / H]];
  // mbarriers: full[3] (package landed), empty[3] (stage free: MMAs done and
  // the state warps read its U~ and decays), sready[2] (S^T stored), xf
  // (X^T ready), uready (U^T stored), accf (acc^T ready), of[2] / oe[2] (O^T
  // ready / read), drain
  const uint32_t bars = sbase + kChMisc;
  const uint32_t full0 = bars, empty0 = bars + 24, sready0 = bars + 48, accf = bars + 64,
                 xf = bars + 72, of0 = bars + 80, oe0 = bars + 96, drain = bars + 112,
                 uready = bars + 120;
  if (tid == 0) {
    for (int s = 0; s < kChStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1 + 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(sready0 + 8 * s, 4);
      mbar_init(sready0 + 88 + 8 * s, 4);  // second channel half (column halves)
      mbar_init(of0 + 8 * s, 1);
      mbar_init(oe0 + 8 * s, 4);
    }
    mbar_init(accf, 1);
    mbar_init(xf, 1);
    mbar_init(uready, 4);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (kHalf && tid == 0) prefetch_tmap(tm_o);
  if (warp == 0) tmem_alloc(bars + 128, 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kChMisc + 128);
  const int N = m.ok ? (m.len + kC - 1) / kC : 0;
  bool failed = false;

  if (warp < 4 && kHalf) {
    failed = !chain_state_half(smem, a, tm_o, u, hv, m, N, tmem, bars);
    if (lane == 0) bulk_wait<0>();  // the output stores are complete before the CTA exits
  } else if (warp < 4) {
    const int j = tid;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int64_t cs = dv;  // stride between channels (rows) of a state
    float S[kDK];
    if (m.ok && m.src >= 0) {
      const float *s0 = a.c.pool + ((int64_t)m.src * H + h) * kDK * dv + j;
#pragma unroll
      for (int c = 0; c < kDK; ++c) S[c] = s0[c * cs];
    } else {
#pragma unroll
      for (int c = 0; c < kDK; ++c) S[c] = 0.f;
    }
    // outputs of chunk n from O^T buffer n & 1: token t of the chunk is
    // column t, thread j holds value column j.  Stored directly: per token,
    // the 128 threads write its 128 contiguous outputs (256 bytes).  Half
    // `hf` (tokens 32 hf .. 32 hf + 31) at a time: the first half goes out
    // while the next chunk's X^T runs on the tensor cores, the second while
    // its acc^T runs; the buffer is handed back after the second.
    auto retire = [&](int n, int hf) -> bool {
      const int b = n & 1;
      if (hf == 0 && !warp_wait(of0 + 8 * b, (n >> 1) & 1)) return false;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32_async(lane_base + 192 + 128 * b + 32 * hf, v);
      tmem_wait_ld();
      reg_fence(v);
      if (hf == 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(oe0 + 8 * b);
      }
      const int cl = min(kC, m.len - n * kC) - 32 * hf;
      const int64_t ts = (int64_t)H * dv;
      __nv_bfloat16 *o = a.c.out + ((int64_t)(m.tok0 + n * kC + 32 * hf) * H + h) * dv + j;
      if (cl >= 32) {
#pragma unroll
        for (int t = 0; t < 32; ++t) o[t * ts] = __float2bfloat16_rn(__uint_as_float(v[t]));
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t < cl) o[t * ts] = __float2bfloat16_rn(__uint_as_float(v[t]));
      }
      return true;
    };
    const int snap_every = a.c.snap_interval > 0 ? a.c.snap_interval / kC : 0;
    int snap_left = snap_every;
    int64_t snap_next = m.snap_off;
    for (int n = 0; n < N; ++n) {
      const int b = n & 1, st = n % kChStages;
      // bf16(S^T) -> TMEM: column q holds channels 2q (low half) and 2q + 1.
      // The last product to read it, chunk n-1's, completed before that
      // chunk's acc^T, which the update of chunk n-1 waited for.
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        uint32_t r[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) r[q] = pack_bf16x2(S[64 * p + 2 * q], S[64 * p + 2 * q + 1]);
        tmem_st32(lane_base + 384 + 32 * p, r);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sready0 + 8 * b);
      if (n > 0 && !retire(n - 1, 0)) { failed = true; break; }
      if (!warp_wait(full0 + 8 * st, (n / kChStages) & 1) || !warp_wait(xf, n & 1)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const uint32_t sp = sbase + st * (uint32_t)kCoopPkgBytes;
      {  // U^T = U~^T - X^T into tensor memory: column q holds tokens 2q (low half), 2q + 1;
         // row j of the package's U~^T holds this thread's 64 tokens
        float x[64];
        tmem_ld64(lane_base + 128 + 128 * b, x);
        uint32_t r[32];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {  // tokens 8 q8 .. 8 q8 + 7
          const uint4 w = ld_shared_v4(sp + kPkU + sw128_chunk(j, q8));
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = 8 * q8 + 2 * e;
            r[4 * q8 + e] = pack_bf16x2(bf16lo(wv[e]) - x[t], bf16hi(wv[e]) - x[t + 1]);
          }
        }
        tmem_st32(lane_base + 448, r);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(uready);
      if (n > 0) retire(n - 1, 1);
      if (!warp_wait(accf, n & 1)) { failed = true; break; }
      tc_fence_after();
      const float4 *egc = reinterpret_cast<const float4 *>(smem + st * kCoopPkgBytes + kPkDec);
#pragma unroll
      for (int p = 0; p < 2; ++p) {  // S = Diag(e^{G_C}) S + acc, 64 channels at a time
        uint32_t v[2][32];
        tmem_ld32_async(lane_base + 64 * p, v[0]);
        tmem_ld32_async(lane_base + 64 * p + 32, v[1]);
        tmem_wait_ld();
        reg_fence(v[0]);
        reg_fence(v[1]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int c = 64 * p + 32 * hh + 4 * q;
            const float4 e = egc[c / 4];
            S[c] = fmaf(e.x, S[c], __uint_as_float(v[hh][4 * q]));
            S[c + 1] = fmaf(e.y, S[c + 1], __uint_as_float(v[hh][4 * q + 1]));
            S[c + 2] = fmaf(e.z, S[c + 2], __uint_as_float(v[hh][4 * q + 2]));
            S[c + 3] = fmaf(e.w, S[c + 3], __uint_as_float(v[hh][4 * q + 3]));
          }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      // a snapshot after every snap_every full chunks (the interval is a
      // multiple of the chunk, so a ragged last chunk never ends on one)
      const int cl = min(kC, m.len - n * kC);
      if (snap_every > 0 && --snap_left == 0 && cl == kC) {
        snap_left = snap_every;
        const int64_t s = snap_next++;
        if (s < a.c.snaps_capacity) {
          float *base =
              snapshot_base(a.c.snaps, a.c.snap_slots, a.c.pool, s, H, h, (int64_t)kDK * dv);
          if (base) {
            float *d = base + j;
#pragma unroll
            for (int c = 0; c < kDK; ++c) d[c * cs] = S[c];
          }
        } else if (j == 0) {
          raise_error(a.c.err, ERR_SNAP_CAPACITY);
        }
      }
    }
    if (!failed && N > 0 && !(retire(N - 1, 0) && retire(N - 1, 1))) failed = true;
    // a unit flagged by a producer keeps its source for the exact recomputation
    const bool flagged =
        atomicAdd(a.c.rerun + u, 0u) == a.epoch;  // (all of its packages are consumed)
    if (!failed && m.ok && !flagged) {
      float *d = a.c.pool + ((int64_t)m.dst * H + h) * kDK * dv + j;
#pragma unroll
      for (int c = 0; c < kDK; ++c) d[c * cs] = S[c];
    }
  } else if (warp == 4 && lane == 0) {
    unsigned long long *consumed = a.consumed + ((size_t)hv * a.units + u) * kCoopRing;
    constexpr int kM = kHalf ? 64 : 128;  // value columns this CTA carries
    bool issued = false;
    for (int n = 0; n < N; ++n) {
      const int b = n & 1, st = n % kChStages;
      const uint32_t sp = sbase + st * (uint32_t)kCoopPkgBytes;
      if (!mbar_wait(full0 + 8 * st, (n / kChStages) & 1)) {
        failed = true;
        break;
      }
      // the package has landed in shared memory (its ring slot has been read
      // in full), so the slot can take another one; nothing of this thread
      // needs ordering before the flag, and a release would stall the MMA
      // issue for an L2 round trip
      st_relaxed_u64(consumed + n % kCoopRing, coop_tag(a.epoch, n));
      if ((n > 1 && !mbar_wait(oe0 + 8 * b, ((n - 2) >> 1) & 1)) ||
          !mbar_wait(sready0 + 8 * b, (n >> 1) & 1)) {
        failed = true;
        break;
      }
      tc_fence_after();
      issued = true;
      const uint32_t xo = tmem + 128 + 128 * b, o = xo + 64, sa = tmem + 384, ut = tmem + 448;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {  // [X^T | O^T] = S^T [W^; Q+']^T: one N = 128 product
        if (kHalf && kk == 4) {  // column halves store S^T a channel half at a time
          if (!mbar_wait(sready0 + 88 + 8 * b, (n >> 1) & 1)) { failed = true; break; }
          tc_fence_after();
        }
        mma_bf16_ts(xo, sa + kk * 8,
                    sw128_desc(sp + kPkWQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                    idesc_bf16(kM, 128, 0, 0), kk > 0);
      }
      if (failed) break;
      mma_commit(xf);
      if (!mbar_wait(uready, n & 1)) { failed = true; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // acc^T = U^T K^
        mma_bf16_ts(tmem, ut + kk * 8, sw128_desc(sp + kPkKm + kk * 2048, 8192, 1024),
                    idesc_bf16(kM, 128, 0, 1), kk > 0);
      mma_commit(accf);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // O^T += U^T M^T
        mma_bf16_ts(o, ut + kk * 8, sw128_desc(sp + kPkM + kk * 32, 16, 1024),
                    idesc_bf16(kM, 64, 0, 0), 1);
      mma_commit(of0 + 8 * b);
      mma_commit(empty0 + 8 * st);
    }
    if (issued) {  // every MMA done before the tensor memory is released
      mma_commit(drain);
      if (!mbar_wait(drain, 0)) failed = true;
    }
  } else if (warp >= 5 && lane == 0) {
    // one loader per package stage: warp 5 + k requests the chunks n = k (mod
    // 3).  A loader's acquire read of its next ready flag stalls it for about
    // the length of a chunk step, so a single loader serialised the chain
    // (2^20-token prefill, measured back to back on one GPU: 21.8 ms with one
    // loader, 19.4 with two; on another GPU 21.1 with two, 19.6 with three).
    // The ready flag of the loader's next package is read (acquire) as soon
    // as this one's copy is requested, so that L2 round trip overlaps the
    // wait for the stage.
    const int k = warp - 5, st = k;
    const unsigned long long *ready = a.ready + u * kCoopRing;
    const uint8_t *ring_u = a.ring + (size_t)u * kCoopRing * kCoopPkgBytes;
    unsigned long long seen = N > k ? ld_acquire_u64(ready + k) : 0ull;
    int issued = -1;  // last chunk whose copy this loader requested
    for (int n = k; n < N; n += kChStages) {
      const unsigned long long want = coop_tag(a.epoch, n);
      if (seen < want && !coop_flag_wait(ready + n % kCoopRing, want, a.hdr + 1)) {
        failed = true;
        break;
      }
      if (n >= kChStages && !mbar_wait(empty0 + 8 * st, ((n - kChStages) / kChStages) & 1)) {
        failed = true;
        break;
      }
      fence_proxy_async_all();  // the package was written by another SM
      const uint8_t *src = ring_u + (size_t)(n % kCoopRing) * kCoopPkgBytes;
      const uint32_t dst = sbase + st * (uint32_t)kCoopPkgBytes, bar = full0 + 8 * st;
      if (kHalf) {  // all but the other column half's rows of U~^T (8 KiB pieces, 1 KiB tail)
        const uint32_t skip = kPkU + 8192u * (1 - hv);
        mbar_expect_tx(bar, (uint32_t)kCoopPkgBytes - 8192u);
        for (uint32_t o = 0; o < (uint32_t)kCoopPkgBytes; o += 8192u)
          if (o != skip)
            bulk_g2s(dst + o, src + o, min(8192u, (uint32_t)kCoopPkgBytes - o), bar);
      } else {
        mbar_expect_tx(bar, (uint32_t)kCoopPkgBytes);
        for (uint32_t q = 0; q < kPkPieces; ++q)
          bulk_g2s(dst + q * kPkPiece, src + q * kPkPiece, kPkPiece, bar);
      }
      issued = n;
      if (n + kChStages < N) seen = ld_acquire_u64(ready + (n + kChStages) % kCoopRing);
    }
    // its last copy lands before the CTA exits (earlier ones landed before
    // their stage was reused)
    if (issued >= 0) mbar_wait(full0 + 8 * st, (issued / kChStages) & 1);
  }
  if (failed) coop_abort(a);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    coop_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                const __grid_constant__ CUtensorMap tm_o, const CoopArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) coop_abort(a);
    return;
  }
  if ((int)blockIdx.x < a.units * a.split) {
    if (a.split == 2)
      coop_chain<true>(smem, a, &tm_o, blockIdx.x % a.units, blockIdx.x / a.units);
    else
      coop_chain<false>(smem, a, &tm_o, blockIdx.x, 0);
  } else {
    coop_producer(smem, &tm_q, &tm_k, &tm_v, &tm_g, a);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D map over a [rows][inner] bf16 array, 64 x 64 boxes, 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows][inner] with unswizzled boxes of 16 columns x 32 rows (one
// warp's outputs of half a chunk in a cooperative chain CTA)
bool make_map_o16(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows][inner] with 128-byte swizzled boxes of 32 columns x 128 rows
// (one (state, 32-column block) per box); false when it cannot be encoded or
// its rows overflow the 32-bit TMA coordinate
bool make_map_f32(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn || !base || rows == 0 || rows >= (1ull << 31)) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DV>
cudaError_t launch_dv(const PrefillPlan &p, const CUtensorMap &mq, const CUtensorMap &mk,
                      const CUtensorMap &mv, const CUtensorMap &mg) {
  constexpr uint32_t smem = Layout<DV>::kBytes;
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void *>(chunked_kernel<DV>), smem);
  if (e != cudaSuccess) return e;
  ChunkArgs a;
  a.beta = static_cast<const __nv_bfloat16 *>(p.beta);
  a.meta = p.meta;
  a.order = p.order;
  a.pool = p.pool;
  a.out = static_cast<__nv_bfloat16 *>(p.out);
  a.snaps = p.snaps;
  a.snap_slots = p.snap_slots;
  a.snaps_capacity = p.snaps_capacity;
  a.snap_interval = p.snap_interval;
  a.H = p.H;
  a.dv = p.dv;
  a.n_dvb = p.dv / DV;
  a.err = p.err;
  a.rerun = p.rerun;
  a.epoch = p.epoch;
  const unsigned grid = (unsigned)((int64_t)p.B * p.H * a.n_dvb);
  CUtensorMap mo, msnap, mpool;
  if (!make_map(&mo, p.out, (uint64_t)p.H * p.dv, (uint64_t)p.T_total)) return cudaErrorInvalidValue;
  std::memset(&msnap, 0, sizeof(msnap));
  std::memset(&mpool, 0, sizeof(mpool));
  const bool snap_ok = p.snaps_capacity > 0 && p.snaps &&
                       make_map_f32(&msnap, p.snaps, (uint64_t)p.dv,
                                    (uint64_t)p.snaps_capacity * p.H * kDK);
  const bool pool_ok = make_map_f32(&mpool, p.pool, (uint64_t)p.dv, (uint64_t)p.n_slots * p.H * kDK);
  a.snap_tma = (p.snap_slots ? pool_ok : snap_ok) ? 1 : 0;
  chunked_kernel<DV><<<grid, kThreads, smem, p.stream>>>(mq, mk, mv, mg, mo, msnap, mpool, a);
  return cudaGetLastError();
}

// Grid of the cooperative kernel on the current device (0 when it cannot run
// there: no cooperative launch, or fewer than 16 producer CTAs would remain
// beside `chains` chain CTAs).
int coop_grid(int chains) {
  if (set_smem_limit_once(reinterpret_cast<const void *>(coop_kernel), kCoopSmem) != cudaSuccess)
    return 0;
  int dev = 0, sms = 0, coop = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, coop_kernel, kThreads, kCoopSmem) !=
          cudaSuccess)
    return 0;
  const int grid = sms * per_sm;
  return grid >= chains + 16 ? grid : 0;
}

// Chunks per cycle the cooperative grid sustains with `split` chain CTAs per
// pair: its producers prepare a chunk each in about kProducerCycles, a chain
// CTA takes kChainCycles (whole columns) or kHalfChainCycles (column halves)
// per chunk of its pair, and the slower side sets the pace (cycle counts
// measured on GB300).
constexpr double kProducerCycles = 15000, kChainCycles = 2900, kHalfChainCycles = 1900;
double coop_rate(int grid, int units, int split) {
  const double producers = grid - units * split;
  return fmin(producers / kProducerCycles,
              units / (split == 2 ? kHalfChainCycles : kChainCycles));
}

cudaError_t launch_coop(const PrefillPlan &p, int grid, int split, const CUtensorMap &mq,
                        const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mg) {
  CoopArgs a;
  a.c.beta = static_cast<const __nv_bfloat16 *>(p.beta);
  a.c.meta = p.meta;
  a.c.order = p.order;
  a.c.pool = p.pool;
  a.c.out = static_cast<__nv_bfloat16 *>(p.out);
  a.c.snaps = p.snaps;
  a.c.snap_slots = p.snap_slots;
  a.c.snaps_capacity = p.snaps_capacity;
  a.c.snap_interval = p.snap_interval;
  a.c.H = p.H;
  a.c.dv = p.dv;
  a.c.n_dvb = 1;
  a.c.err = p.err;
  a.c.rerun = p.rerun;
  a.c.epoch = p.epoch;
  a.c.snap_tma = 0;  // the chain CTAs store snapshots directly (coalesced columns)
  a.units = p.B * p.H;
  a.split = split;
  a.ring = p.coop_ring;
  a.ready = p.coop_flags;
  a.consumed = p.coop_flags + (size_t)a.units * kCoopRing;
  a.hdr = p.coop_hdr;
  a.epoch = p.epoch;
  CUtensorMap q = mq, k = mk, v = mv, g = mg, o;
  if (!make_map_o16(&o, p.out, (uint64_t)p.H * p.dv, (uint64_t)p.T_total)) return cudaErrorInvalidValue;
  void *args[] = {&q, &k, &v, &g, &o, &a};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(coop_kernel), dim3(grid),
                                     dim3(kThreads), args, kCoopSmem, p.stream);
}

}  // namespace

bool chunked_supported(const PrefillPlan &p) {
  return p.dtype == KDA_BF16 && p.dk == 128 && (p.dv == 128 || p.dv == 64) && p.T_total > 0 &&
         (p.snap_interval % kC) == 0 && encode_fn() != nullptr;
}

bool coop_supported(const PrefillPlan &p) {
  return chunked_supported(p) && p.dv == 128 && p.coop_ring != nullptr &&
         (int64_t)p.B * p.H <= kCoopMaxUnits && coop_grid(p.B * p.H) > 0;
}

bool coop_halves_supported(const PrefillPlan &p) {
  return coop_supported(p) && coop_grid(2 * p.B * p.H) > 0;
}

cudaError_t launch_chunked_prefill(const PrefillPlan &p, int mode) {
  CUtensorMap mq, mk, mv, mg;
  const uint64_t T = (uint64_t)p.T_total;
  if (!make_map(&mq, p.q, (uint64_t)p.H * kDK, T) || !make_map(&mk, p.k, (uint64_t)p.H * kDK, T) ||
      !make_map(&mv, p.v, (uint64_t)p.H * p.dv, T) || !make_map(&mg, p.g, (uint64_t)p.H * kDK, T))
    return cudaErrorInvalidValue;
  // cooperative producer/chain grid when few (sequence, head) pairs would
  // leave most SMs idle; otherwise one CTA per (sequence, head, dv block)
  if (mode == kChunkCoop) return launch_coop(p, coop_grid(p.B * p.H), 1, mq, mk, mv, mg);
  if (mode == kChunkCoopHalves) return launch_coop(p, coop_grid(2 * p.B * p.H), 2, mq, mk, mv, mg);
  if (mode == kChunkAuto && coop_supported(p)) {
    // column halves when their faster chains outweigh the producers they take
    const int units = p.B * p.H, g1 = coop_grid(units), g2 = coop_grid(2 * units);
    const bool halves = g2 > 0 && coop_rate(g2, units, 2) > coop_rate(g1, units, 1);
    return launch_coop(p, halves ? g2 : g1, halves ? 2 : 1, mq, mk, mv, mg);
  }
  // Two 64-column dv blocks per (sequence, head) only while they all fit in
  // one wave (one CTA per SM): a 64-column CTA is about 13% faster than a
  // 128-column one on the same chunks, so a second wave costs more than the
  // narrower blocks gain (3 x 32768 tokens x 32 heads: 6.78 ms with 192
  // narrow CTAs, 3.90 ms with 96 wide ones, back to back on one GPU).
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  const bool narrow = 2 * (int64_t)p.B * p.H <= sms && p.dv == 128;
  if (p.dv == 64 || narrow) return launch_dv<64>(p, mq, mk, mv, mg);
  return launch_dv<128>(p, mq, mk, mv, mg);
}

}  // namespace kda
