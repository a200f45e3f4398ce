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
//   prep  cumulative decay per channel, K+, Q+, K- (in place), K_end, S0'
//   MMA1  [K+; Q+] K-^T                 M=128 N=64  K=128  -> A, Q+K-^T (TMEM)
//   solve T = (I + A)^{-1} Diag(beta)    fp32, 16x16 blocks, CUDA cores
//   MMA2  [T; M] K+ and [T; M] V        -> W, U~ (TMEM)
//   MMA3  U~ -= W S0'  ;  O = Q+ S0'
//   MMA4  K_end^T U    ;  O += M U
//   out   o rows -> global bf16; S = Diag(e^{G_C}) S + K_end^T U (registers),
//         snapshot / final state -> global fp32
// All MMAs are M = 128 (rows 64..127 of the 64-row operands are ignored).
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
  static constexpr uint32_t kW = kTM + 16384;          // W halves; fp32 L during the solve
  static constexpr uint32_t kU = kW + 16384;           // U halves; fp32 X during the solve
  static constexpr uint32_t kKE = kU + 16384;          // K_end halves
  static constexpr uint32_t kS0 = kKE + 16384;         // S0' halves (128 rows each)
  static constexpr uint32_t kMisc = kS0 + (DV / 64) * 16384;
  static constexpr uint32_t kBars = 0;                 // tma[2], mma
  static constexpr uint32_t kSlot = 24;                // TMEM base address
  static constexpr uint32_t kBeta = 64;                // f32[64]
  static constexpr uint32_t kEgc = kBeta + 256;        // f32[128] e^{G_C}
  static constexpr uint32_t kPart = kEgc + 512;        // f32[2][128] half-chunk decay sums
  static constexpr uint32_t kBytes = kMisc + kPart + 1024;
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
  int64_t snaps_capacity;
  int32_t snap_interval;
  int32_t H, dv, n_dvb;
  uint32_t *err;
};

// A CTA-uniform bounded wait: false (for every thread) if any thread gave up.
__device__ __forceinline__ bool cta_wait(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return !__syncthreads_or(!ok);
}

__device__ __forceinline__ float bf(const uint8_t *base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(base + off));
}
__device__ __forceinline__ void st_bf(uint8_t *base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(x);
}

// Fp32 64x64 unit-lower-triangular system L = I + A with A stored rotated
// (element (r, i) at r*64 + ((i + r) & 63), conflict-free row writes).
__device__ __forceinline__ float Lrot(const float *L, int r, int i) {
  return L[r * 64 + ((i + r) & 63)];
}

// X = (I + A)^{-1} by 16x16 blocks: diagonal blocks by forward substitution,
// then the three bands below the diagonal, X_ab = -X_aa sum_{b<=c<a} A_ac X_cb.
__device__ __forceinline__ void solve_unit_lower(const float *L, float *X, float *Y, int tid) {
  if (tid < 64) {
    const int base = (tid >> 4) * 16, jj = tid & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = (r == jj) ? 1.f : 0.f;
#pragma unroll
      for (int i = 0; i < r; ++i) acc = fmaf(-Lrot(L, base + r, base + i), x[i], acc);
      x[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) X[(base + r) * 64 + base + jj] = x[r];
  }
  __syncthreads();
#pragma unroll 1
  for (int d = 1; d < 4; ++d) {
    const int nblk = 4 - d;
    for (int e = tid; e < nblk * 256; e += kThreads) {
      const int b = e >> 8, r = (e >> 4) & 15, j = e & 15, a = b + d;
      float acc = 0.f;
      for (int c = b; c < a; ++c) {
#pragma unroll
        for (int k = 0; k < 16; ++k)
          acc = fmaf(Lrot(L, 16 * a + r, 16 * c + k), X[(16 * c + k) * 64 + 16 * b + j], acc);
      }
      Y[e] = acc;
    }
    __syncthreads();
    for (int e = tid; e < nblk * 256; e += kThreads) {
      const int b = e >> 8, r = (e >> 4) & 15, j = e & 15, a = b + d;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        acc = fmaf(X[(16 * a + r) * 64 + 16 * a + k], Y[b * 256 + k * 16 + j], acc);
      X[(16 * a + r) * 64 + 16 * b + j] = -acc;
    }
    __syncthreads();
  }
}

template <int DV>
__global__ void __launch_bounds__(kThreads, 1)
    chunked_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                   const ChunkArgs a) {
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
  float *s_egc = reinterpret_cast<float *>(misc + Ly::kEgc);
  float *s_part = reinterpret_cast<float *>(misc + Ly::kPart);

  if (tid == 0) {
    mbar_init(bar_tma0, 1);
    mbar_init(bar_tma0 + 8, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_g);
  }
  if (warp == 0) tmem_alloc(sbase + Ly::kMisc + Ly::kSlot, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(misc + Ly::kSlot);
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);

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
  if (tid == 0 && nchunks > 0) issue_tma(0);
  tma_pending[0] = nchunks > 0;

  const uint32_t idesc_am = idesc_bf16(128, 64, 0, 0);
  const uint32_t idesc_w = idesc_bf16(128, 128, 0, 1);
  const uint32_t idesc_v = idesc_bf16(128, DV, 0, 1);
  const uint32_t idesc_vneg = idesc_bf16(128, DV, 0, 1, 1);
  const uint32_t idesc_ke = idesc_bf16(128, DV, 1, 1);

#pragma unroll 1
  for (int n = 0; n < nchunks; ++n) {
    const int st = n & 1;
    uint8_t *stage = smem + st * Ly::kStage;
    const uint32_t sb = sbase + st * Ly::kStage;
    const int t0 = m.tok0 + n * kC;
    const int cl = min(kC, m.len - n * kC);

    if (n + 1 < nchunks) {
      if (tid == 0) issue_tma(n + 1);
      tma_pending[(n + 1) & 1] = true;
      tma_parity[(n + 1) & 1] = ((n + 1) >> 1) & 1;
    }
    if (!cta_wait(bar_tma0 + 8 * st, (n >> 1) & 1)) { aborted = true; break; }
    tma_pending[st] = false;

    // ------------------------------------------------------------ prep
    const int ch = tid & 127, hf = tid >> 7;
    const uint32_t kq_half = (ch >> 6) * 16384, g_half = (ch >> 6) * 8192;
    const int cc = ch & 63;
    {
      float s = 0.f;
      for (int r = 32 * hf; r < 32 * hf + 32 && r < cl; ++r)
        s += bf(stage, Ly::kG + g_half + sw128_offset(r, cc));
      s_part[hf * 128 + ch] = s;
      if (tid < 64)
        s_beta[tid] = tid < cl ? __bfloat162float(a.beta[(int64_t)(t0 + tid) * H + h]) : 0.f;
      if (cl < kC) {  // ragged tail: zero the v rows past the sequence end
        for (int e = tid; e < (kC - cl) * (DV / 8); e += kThreads) {
          const int r = cl + e / (DV / 8), chk = e % (DV / 8);
          st_shared_v4(sb + Ly::kV + (chk >> 3) * 8192 + sw128_chunk(r, chk & 7), 0, 0, 0, 0);
        }
      }
    }
    __syncthreads();
    {
      const float p0 = s_part[ch], p1 = s_part[128 + ch];
      const float cke = expf(p1);  // e^{G_C - a}
      if (hf == 0) s_egc[ch] = expf(p0 + p1);
      float x = 0.f;
      for (int it = 0; it < 32; ++it) {
        const int r = hf ? 32 + it : 31 - it;
        const uint32_t okq = kq_half + sw128_offset(r, cc);
        const uint32_t og = Ly::kG + g_half + sw128_offset(r, cc);
        const uint32_t oke = Ly::kKE + g_half + sw128_offset(r, cc);
        float gr = 0.f;
        if (r < cl) gr = bf(stage, og);
        if (hf) x += gr;  // x = G_r - a
        if (r < cl) {
          const float kv = bf(stage, okq), qv = bf(stage, Ly::kQ + okq);
          const float e1 = __expf(x), e2 = __expf(-x);
          st_bf(stage, okq, kv * e1);
          st_bf(stage, Ly::kQ + okq, qv * e1);
          st_bf(stage, og, kv * e2);
          st_bf(smem, oke, kv * e2 * cke);
        } else {
          st_bf(stage, okq, 0.f);
          st_bf(stage, Ly::kQ + okq, 0.f);
          st_bf(stage, og, 0.f);
          st_bf(smem, oke, 0.f);
        }
        if (!hf) x -= gr;
      }
      // S0' = Diag(e^{a}) S as the bf16 operand (MN-major: row = channel c)
      const float ea = expf(s_part[c]);
#pragma unroll
      for (int j = 0; j < NH / 8; ++j) {
        const int col = col0 + 8 * j;
        st_shared_v4(sbase + Ly::kS0 + (col >> 6) * 16384 + sw128_chunk(c, (col & 63) >> 3),
                     pack_bf16x2(ea * S[8 * j], ea * S[8 * j + 1]),
                     pack_bf16x2(ea * S[8 * j + 2], ea * S[8 * j + 3]),
                     pack_bf16x2(ea * S[8 * j + 4], ea * S[8 * j + 5]),
                     pack_bf16x2(ea * S[8 * j + 6], ea * S[8 * j + 7]));
      }
    }
    fence_async_smem();
    __syncthreads();

    // ------------------------------------------------------------ MMA1
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = sw128_desc(sb + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = sw128_desc(sb + Ly::kG + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
        mma_bf16(tmem + 256, ad, bd, idesc_am, kk > 0);
      }
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!cta_wait(bar_mma, mma_phase)) { aborted = true; break; }
    mma_phase ^= 1;
    mma_pending = false;
    tc_fence_after();

    // A (rows 0..63) into the fp32 system; M (rows 64..127) into [T; M]
    float *Lm = reinterpret_cast<float *>(smem + Ly::kW);
    float *Xm = reinterpret_cast<float *>(smem + Ly::kU);
    float *Ym = reinterpret_cast<float *>(stage + Ly::kG);
    {
      float v[32];
      tmem_ld32(lane_base + 256 + colhalf * 32, v);
      const int rr = quarter * 32 + lane;
      if (quarter < 2) {
        const float br = s_beta[rr];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = colhalf * 32 + j;
          Lm[rr * 64 + ((i + rr) & 63)] = (i < rr) ? br * v[j] : 0.f;
        }
      } else {
        const int r = rr - 64;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float w8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = colhalf * 32 + q4 * 8 + j;
            w8[j] = (i <= r) ? v[q4 * 8 + j] : 0.f;
          }
          st_shared_v4(sbase + Ly::kTM + sw128_chunk(64 + r, colhalf * 4 + q4),
                       pack_bf16x2(w8[0], w8[1]), pack_bf16x2(w8[2], w8[3]),
                       pack_bf16x2(w8[4], w8[5]), pack_bf16x2(w8[6], w8[7]));
        }
      }
    }
    tc_fence_before();
    __syncthreads();

    // ------------------------------------------------------------ solve
    solve_unit_lower(Lm, Xm, Ym, tid);
    {
      const int r = tid >> 2, q4 = tid & 3;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float t8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int col = q4 * 16 + half * 8 + j;
          t8[j] = (col <= r) ? Xm[r * 64 + col] * s_beta[col] : 0.f;
        }
        st_shared_v4(sbase + Ly::kTM + sw128_chunk(r, q4 * 2 + half), pack_bf16x2(t8[0], t8[1]),
                     pack_bf16x2(t8[2], t8[3]), pack_bf16x2(t8[4], t8[5]),
                     pack_bf16x2(t8[6], t8[7]));
      }
    }
    fence_async_smem();
    __syncthreads();

    // ------------------------------------------------------------ MMA2
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = sw128_desc(sbase + Ly::kTM + kk * 32, 16, 1024);
        mma_bf16(tmem + 0, ad, sw128_desc(sb + kk * 2048, 16384, 1024), idesc_w, kk > 0);
        mma_bf16(tmem + 128, ad, sw128_desc(sb + Ly::kV + kk * 2048, 8192, 1024), idesc_v, kk > 0);
      }
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!cta_wait(bar_mma, mma_phase)) { aborted = true; break; }
    mma_phase ^= 1;
    mma_pending = false;
    tc_fence_after();

    // W (rows 0..63) -> bf16 K-major operand
    if (quarter < 2) {
      const int r = quarter * 32 + lane;
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        float v[32];
        tmem_ld32(lane_base + colhalf * 64 + p * 32, v);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(sbase + Ly::kW + colhalf * 8192 + sw128_chunk(r, p * 4 + q4),
                       pack_bf16x2(v[q4 * 8], v[q4 * 8 + 1]), pack_bf16x2(v[q4 * 8 + 2], v[q4 * 8 + 3]),
                       pack_bf16x2(v[q4 * 8 + 4], v[q4 * 8 + 5]),
                       pack_bf16x2(v[q4 * 8 + 6], v[q4 * 8 + 7]));
      }
    }
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
        mma_bf16(tmem + 384,
                 sw128_desc(sb + Ly::kQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), bd,
                 idesc_v, kk > 0);
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
#pragma unroll
      for (int p = 0; p < NH / 32; ++p) {
        float v[32];
        tmem_ld32(lane_base + 128 + col0 + p * 32, v);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int col = col0 + p * 32 + q4 * 8;
          st_shared_v4(sbase + Ly::kU + (col >> 6) * 8192 + sw128_chunk(r, (col & 63) >> 3),
                       pack_bf16x2(v[q4 * 8], v[q4 * 8 + 1]), pack_bf16x2(v[q4 * 8 + 2], v[q4 * 8 + 3]),
                       pack_bf16x2(v[q4 * 8 + 4], v[q4 * 8 + 5]),
                       pack_bf16x2(v[q4 * 8 + 6], v[q4 * 8 + 7]));
        }
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
        mma_bf16(tmem + 256, sw128_desc(sbase + Ly::kKE + kk * 2048, 8192, 1024), bd, idesc_ke,
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
    if (quarter < 2) {
      const int r = quarter * 32 + lane;
      __nv_bfloat16 *orow = a.out + ((int64_t)(t0 + r) * H + h) * dv + dv0 + col0;
#pragma unroll
      for (int p = 0; p < NH / 32; ++p) {
        float v[32];
        tmem_ld32(lane_base + 384 + col0 + p * 32, v);
        if (r < cl) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + p * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            dst[q4] = make_uint4(pack_bf16x2(v[q4 * 8], v[q4 * 8 + 1]),
                                 pack_bf16x2(v[q4 * 8 + 2], v[q4 * 8 + 3]),
                                 pack_bf16x2(v[q4 * 8 + 4], v[q4 * 8 + 5]),
                                 pack_bf16x2(v[q4 * 8 + 6], v[q4 * 8 + 7]));
        }
      }
    }
    {
      const float egc = s_egc[c];
#pragma unroll
      for (int p = 0; p < NH / 32; ++p) {
        float v[32];
        tmem_ld32(lane_base + 256 + col0 + p * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) S[p * 32 + j] = fmaf(egc, S[p * 32 + j], v[j]);
      }
      const int64_t done = (int64_t)n * kC + cl;
      if (a.snap_interval > 0 && done % a.snap_interval == 0) {
        const int64_t s = m.snap_off + done / a.snap_interval - 1;
        if (s < a.snaps_capacity) {
          float4 *dst = reinterpret_cast<float4 *>(
              a.snaps + (((s * H + h) * kDK + c) * dv) + dv0 + col0);
#pragma unroll
          for (int j = 0; j < NH / 4; ++j)
            dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
        } else if (tid == 0) {
          raise_error(a.err, ERR_SNAP_CAPACITY);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (aborted) {
    if (tid == 0) raise_error(a.err, ERR_TIMEOUT);
    // drain what is still in flight (bounded), then release TMEM
    for (int s = 0; s < 2; ++s)
      if (tma_pending[s]) mbar_wait(bar_tma0 + 8 * s, tma_parity[s]);
    if (mma_pending) mbar_wait(bar_mma, mma_phase);
  } else {
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

template <int DV>
cudaError_t launch_dv(const PrefillPlan &p, const CUtensorMap &mq, const CUtensorMap &mk,
                      const CUtensorMap &mv, const CUtensorMap &mg) {
  constexpr uint32_t smem = Layout<DV>::kBytes;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(chunked_kernel<DV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  ChunkArgs a;
  a.beta = static_cast<const __nv_bfloat16 *>(p.beta);
  a.meta = p.meta;
  a.order = p.order;
  a.pool = p.pool;
  a.out = static_cast<__nv_bfloat16 *>(p.out);
  a.snaps = p.snaps;
  a.snaps_capacity = p.snaps_capacity;
  a.snap_interval = p.snap_interval;
  a.H = p.H;
  a.dv = p.dv;
  a.n_dvb = p.dv / DV;
  a.err = p.err;
  const unsigned grid = (unsigned)((int64_t)p.B * p.H * a.n_dvb);
  chunked_kernel<DV><<<grid, kThreads, smem, p.stream>>>(mq, mk, mv, mg, a);
  return cudaGetLastError();
}

}  // namespace

bool chunked_supported(const PrefillPlan &p) {
  return p.dtype == KDA_BF16 && p.dk == 128 && (p.dv == 128 || p.dv == 64) && p.T_total > 0 &&
         (p.snap_interval % kC) == 0 && encode_fn() != nullptr;
}

cudaError_t launch_chunked_prefill(const PrefillPlan &p) {
  CUtensorMap mq, mk, mv, mg;
  const uint64_t T = (uint64_t)p.T_total;
  if (!make_map(&mq, p.q, (uint64_t)p.H * kDK, T) || !make_map(&mk, p.k, (uint64_t)p.H * kDK, T) ||
      !make_map(&mv, p.v, (uint64_t)p.H * p.dv, T) || !make_map(&mg, p.g, (uint64_t)p.H * kDK, T))
    return cudaErrorInvalidValue;
  // one dv block of 128 per (sequence, head) when that fills the GPU, else 64
  const bool narrow = (int64_t)p.B * p.H < 148 && p.dv == 128;
  if (p.dv == 64 || narrow) return launch_dv<64>(p, mq, mk, mv, mg);
  return launch_dv<128>(p, mq, mk, mv, mg);
}

}  // namespace kda
