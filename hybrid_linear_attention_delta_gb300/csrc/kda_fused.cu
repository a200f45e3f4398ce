// kda_fused.cu -- the layer around the KDA recurrence that a serving stack
// runs with it: a short causal convolution of the raw q, k, v channels, whose
// last inputs are kept per slot beside the matrix state, and the gated
// RMSNorm of the outputs.
//
// "Kimi K3 + vLLM: Inside the Day-0 Production Integration": a KDA layer keeps
// "a short causal convolution state" beside its matrix state ("Kimi Delta
// Attention: When Prefix Caching Meets Recurrent State"), and its fused decode
// kernel folds the causal convolution, the recurrent state update, the gating
// and the RMSNorm into one launch ("Separate Prefill/Decode Code Paths"); the
// vLLM recipe page for Kimi-K3 fuses the output RMSNorm and its sigmoid gate
// into one kernel.  Per token t and head h, with W = 4 taps per channel:
//     [q~ | k~ | v~]_t = act(sum_i w[c][i] x[t - (W-1) + i][c])   (raw x, causal)
//     q = q~ / |q~| / sqrt(dk),  k = k~ / |k~|,  v = v~             (then the recurrence)
//     y_t = o_t / sqrt(mean(o_t^2) + eps) * w_norm * sigmoid(gate_t)
// Decode runs all of it in one kernel (decode_fused_kernel).  Prefill runs it
// around the chunked kernels: conv_prefill_kernel writes q, k, v for the
// batch, conv_state_kernel the new convolution states, and rms_gate_kernel
// turns the prefill's outputs into y.  Reductions (L2 norms, RMS) run in a
// fixed order: results are deterministic.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kMaxConvC = 384;    // channels of a head: 2 dk + dv <= 384

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }
// the gate of the prefill's output norm, one per output element: the fast
// exponential and division intrinsics (relative error a few ulp, far inside
// the output's bf16 rounding); 0 for x below about -88, where e^-x overflows
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float act_f(float y, int act) {
  return act == 1 ? y / (1.f + expf(-y)) : y;
}

template <typename T>
__device__ __forceinline__ float raw_input(const FusedParams &f, int64_t t, int H, int h, int dk,
                                           int dv, int c) {
  if (c < dk) return to_f32(static_cast<const T *>(f.xq)[(t * H + h) * dk + c]);
  if (c < 2 * dk) return to_f32(static_cast<const T *>(f.xk)[(t * H + h) * dk + c - dk]);
  return to_f32(static_cast<const T *>(f.xv)[(t * H + h) * dv + c - 2 * dk]);
}

// Sequence of packed token t: the largest b with cu[b] <= t (cu validated by
// the plan kernel; empty sequences are skipped by taking the largest).
__device__ __forceinline__ int seq_of(const int32_t *cu, int B, int64_t t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Four consecutive elements of T as one vector (8 bytes for bf16, 16 for
// fp32), and their conversion to and from fp32 (round to nearest even).
template <typename T> struct Quad;
template <> struct Quad<__nv_bfloat16> { uint2 u; };
template <> struct Quad<float> { uint4 u; };

template <typename T>
__device__ __forceinline__ Quad<T> load_quad(const T *p) {
  Quad<T> q;
  q.u = __ldcs(reinterpret_cast<const decltype(q.u) *>(p));
  return q;
}

__device__ __forceinline__ void unpack_quad(const Quad<__nv_bfloat16> &q, float (&x)[4]) {
  x[0] = __uint_as_float(q.u.x << 16);
  x[1] = __uint_as_float(q.u.x & 0xffff0000u);
  x[2] = __uint_as_float(q.u.y << 16);
  x[3] = __uint_as_float(q.u.y & 0xffff0000u);
}
__device__ __forceinline__ void unpack_quad(const Quad<float> &q, float (&x)[4]) {
  x[0] = __uint_as_float(q.u.x); x[1] = __uint_as_float(q.u.y);
  x[2] = __uint_as_float(q.u.z); x[3] = __uint_as_float(q.u.w);
}

__device__ __forceinline__ void store_quad(__nv_bfloat16 *p, const float (&y)[4]) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]), hi = __floats2bfloat162_rn(y[2], y[3]);
  *reinterpret_cast<uint2 *>(p) =
      make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}
__device__ __forceinline__ void store_quad(float *p, const float (&y)[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(y[0], y[1], y[2], y[3]);
}

// The prefill convolution.  A unit is (head h, run of kConvRun consecutive
// packed tokens); a CTA takes kConvUnits units, heads fastest, so the CTAs
// that run together read whole token rows.  Unit u has three warps, one per
// part (q, k, v); lane i owns channels [4 i, 4 i + 4) of the part (one vector
// load per token), so |q~| and |k~| of a token are a shuffle tree inside one
// warp.  A lane keeps its taps and its channels' last three raw inputs in
// registers and walks its run a batch of tokens at a time (64 bytes a lane),
// the batch's loads issued together.  At a run start inside a sequence the
// history is the three tokens before it; at a sequence start, the sequence's
// starting convolution state (zeros without one).  Writes q, k, v (the
// recurrence's inputs) for tokens of sequences the plan accepted.
constexpr int kConvRun = 64;
constexpr int kConvUnits = 2;
constexpr int kConvThreads = 32 * 3 * kConvUnits;
constexpr int kConvBatchBytes = 64;  // per lane in flight: 8 bf16 or 4 fp32 tokens

template <typename T>
__global__ void __launch_bounds__(kConvThreads, 4) conv_prefill_kernel(PrefillPlan p, FusedParams f) {
  constexpr int kConvBatch = kConvBatchBytes / (int)sizeof(Quad<T>);
  const int H = p.H, dk = p.dk, dv = p.dv, C = 2 * dk + dv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = warp / 3, part = warp % 3;  // part 0: q, 1: k, 2: v
  const int dpart = part == 2 ? dv : dk;
  const bool active = 4 * lane < dpart;
  const int64_t u = (int64_t)blockIdx.x * kConvUnits + unit;
  const int h = (int)(u % H);
  if (u / H * kConvRun >= p.T_total) return;  // the whole warp (one unit)
  const int tb = (int)(u / H) * kConvRun;      // token indices fit int32 (T_total does)
  const int te = tb + min(kConvRun, p.T_total - tb);
  const int q4 = active ? 4 * lane : 0;  // first channel of the lane within its part
  const int c0 = part * dk + q4;         // ... within [q | k | v]
  const T *x = static_cast<const T *>(part == 0 ? f.xq : part == 1 ? f.xk : f.xv);
  T *y_out = static_cast<T *>(const_cast<void *>(part == 0 ? p.q : part == 1 ? p.k : p.v));
  const int col = h * dpart + q4, row_stride = H * dpart;

  float w[4][kConvW];
  {
    const float *wp = f.conv_w + ((int64_t)h * C + c0) * kConvW;
    if ((reinterpret_cast<uintptr_t>(f.conv_w) & 15u) == 0) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 t4 = reinterpret_cast<const float4 *>(wp)[e];
        w[e][0] = t4.x; w[e][1] = t4.y; w[e][2] = t4.z; w[e][3] = t4.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int i = 0; i < kConvW; ++i) w[e][i] = wp[e * kConvW + i];
    }
  }

  int b = seq_of(p.cu_seqlens, p.B, tb);
  int start = p.cu_seqlens[b], end = p.cu_seqlens[b + 1];
  int ok = p.meta[b].ok;
  float hist[kConvW - 1][4];
  // the kConvW - 1 raw inputs before token t of sequence b: tokens of the
  // sequence, else its starting convolution state, else zeros
  auto init_hist = [&](int t) {
    const int src = p.meta[b].src;
    const T *cp = static_cast<const T *>(f.conv_pool) +
                  (((int64_t)(src >= 0 ? src : 0) * H + h) * C + c0) * (kConvW - 1);
#pragma unroll
    for (int i = 0; i < kConvW - 1; ++i) {
      const int pos = t - (kConvW - 1) + i;
      if (pos >= start) {
        unpack_quad(load_quad(x + (int64_t)pos * row_stride + col), hist[i]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          hist[i][e] = src >= 0 ? to_f32(cp[e * (kConvW - 1) + (kConvW - 1) + (pos - start)]) : 0.f;
      }
    }
  };
  init_hist(tb);
  const float qscale = rsqrtf((float)dk);

  // one token: convolution, |q~| or |k~| (a shuffle tree over the warp's
  // active lanes; the others hold 0), scaling, store
  auto step = [&](const Quad<T> &xq4, T *dst) {
    float xv[4], y[4], ss = 0.f;
    unpack_quad(xq4, xv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float acc = w[e][kConvW - 1] * xv[e];
#pragma unroll
      for (int i = 0; i < kConvW - 1; ++i) acc = fmaf(w[e][i], hist[i][e], acc);
      y[e] = act_f(acc, f.act);
      ss = fmaf(y[e], y[e], ss);
    }
#pragma unroll
    for (int i = 0; i + 1 < kConvW - 1; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) hist[i][e] = hist[i + 1][e];
#pragma unroll
    for (int e = 0; e < 4; ++e) hist[kConvW - 2][e] = xv[e];
    if (part < 2) {
      if (!active) ss = 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float scale = ss > 0.f ? rsqrtf(ss) : 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) y[e] = part == 0 ? y[e] * scale * qscale : y[e] * scale;
    }
    if (active && ok) store_quad(dst, y);
  };

  // batches inside one sequence issue their loads together; a batch that
  // reaches the run's end or a sequence start goes token by token
  for (int t0 = tb; t0 < te; t0 += kConvBatch) {
    if (t0 + kConvBatch <= te && t0 + kConvBatch <= end) {
      const int64_t off = (int64_t)t0 * row_stride + col;
      Quad<T> xr[kConvBatch];
#pragma unroll
      for (int j = 0; j < kConvBatch; ++j) xr[j] = load_quad(x + off + j * row_stride);
#pragma unroll
      for (int j = 0; j < kConvBatch; ++j) step(xr[j], y_out + off + j * row_stride);
    } else {
      const int t1 = min(t0 + kConvBatch, te);
#pragma unroll 1
      for (int t = t0; t < t1; ++t) {
        if (t >= end) {  // the next sequence (skipping empty ones) starts here
          while (t >= end) {
            ++b;
            start = p.cu_seqlens[b];
            end = p.cu_seqlens[b + 1];
          }
          ok = p.meta[b].ok;
          init_hist(t);
        }
        const int64_t off = (int64_t)t * row_stride + col;
        step(load_quad(x + off), y_out + off);
      }
    }
  }
}

// One CTA per (sequence, head); thread c: channel c.  The new state of a
// channel is the last kConvW - 1 raw inputs of [old state; sequence], read
// before anything is written (so src == dst extends in place).
template <typename T>
__global__ void __launch_bounds__(kMaxConvC) conv_state_kernel(PrefillPlan p, FusedParams f) {
  const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x, H = p.H, dk = p.dk, dv = p.dv;
  const int C = 2 * dk + dv;
  const SeqMeta m = p.meta[b];
  if (!m.ok || c >= C) return;
  T *cp = static_cast<T *>(f.conv_pool);
  float ns[kConvW - 1];
#pragma unroll
  for (int i = 0; i < kConvW - 1; ++i) {
    const int64_t pos = (int64_t)m.len - (kConvW - 1) + i;
    if (pos >= 0)
      ns[i] = raw_input<T>(f, (int64_t)m.tok0 + pos, H, h, dk, dv, c);
    else if (m.src >= 0)
      ns[i] = to_f32(cp[(((int64_t)m.src * H + h) * C + c) * (kConvW - 1) + (kConvW - 1 + pos)]);
    else
      ns[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < kConvW - 1; ++i)
    cp[(((int64_t)m.dst * H + h) * C + c) * (kConvW - 1) + i] = from_f32<T>(ns[i]);
}

// y = o / rms(o) * w * sigmoid(gate) per (token, head) row of dv outputs.
// One warp takes kRmsRows consecutive rows, lane i elements [E i, E i + E)
// of each (E = max(dv / 32, 1): one vector load per row and tensor; lanes
// past dv idle), and issues all their loads before it reduces.  The rows' sequences come from one search
// and a forward walk; rows of sequences the plan did not accept are not
// written.
constexpr int kRmsRows = 4;

template <typename T, int E>
struct alignas(E * sizeof(T)) VecT {
  T x[E];
};

template <typename T, int E>
__global__ void __launch_bounds__(256) rms_gate_kernel(PrefillPlan p, FusedParams f, const T *o,
                                                       T *out) {
  using V = VecT<T, E>;
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRmsRows;
  const int H = p.H, dv = p.dv;
  const int64_t rows = (int64_t)p.T_total * H;
  if (row0 >= rows) return;
  const bool act = E * lane < dv;
  const int col = act ? E * lane : 0;
  const T *gate = static_cast<const T *>(f.gate);
  V v[kRmsRows], gt[kRmsRows];
#pragma unroll
  for (int r = 0; r < kRmsRows; ++r) {
    const int64_t row = row0 + r < rows ? row0 + r : rows - 1;
    v[r] = *reinterpret_cast<const V *>(o + row * dv + col);
    gt[r] = *reinterpret_cast<const V *>(gate + row * dv + col);
  }
  float nw[E];
#pragma unroll
  for (int e = 0; e < E; ++e) nw[e] = f.norm_w[col + e];
  // token and head of the first row (one division a warp), then stepped
  int t = (int)(row0 / H), hh = (int)(row0 - (int64_t)t * H);
  int b = seq_of(p.cu_seqlens, p.B, t);
#pragma unroll
  for (int r = 0; r < kRmsRows; ++r) {
    const int64_t row = row0 + r;
    if (row >= rows) break;
    if (r > 0 && ++hh == H) {
      hh = 0;
      ++t;
    }
    while (b + 1 < p.B && p.cu_seqlens[b + 1] <= t) ++b;
    float x[E], ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] = act ? to_f32(v[r].x[e]) : 0.f;
      ss = fmaf(x[e], x[e], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (!act || !p.meta[b].ok) continue;
    const float rr = rsqrtf(ss / (float)dv + f.eps);
    V y;
#pragma unroll
    for (int e = 0; e < E; ++e) y.x[e] = from_f32<T>(x[e] * rr * nw[e] * sigmoid_fast(to_f32(gt[r].x[e])));
    *reinterpret_cast<V *>(out + row * dv + col) = y;
  }
}

// ------------------------------------------------------------------ decode
// One CTA of 256 threads per (sequence, head), dk = dv = 128; the state
// layout of the 128 x 128 decode kernels (warp w: rows [16 w, +16), lane l:
// columns [4 l, +4)), read once and written once.  The state loads are issued
// first; everything else overlaps them.  Thread c owns raw channel c (q for
// c < 128, k otherwise) and, for c < 128, channel 256 + c (v): its last three raw
// inputs live in registers and go back to the slot's convolution state at the
// end.  Per token: the convolution, the L2
// normalisation of q and k, their rounding to the call's element type (the
// type every call's recurrence takes them in), the recurrence step and the
// gated RMSNorm of the output, with five block barriers.
constexpr int kD = 128;
constexpr int kDecThreads = 256;
constexpr int kRows = kD / (kDecThreads / 32);  // 16
constexpr int kC3 = 3 * kD;                     // channels q | k | v

template <typename T>
__global__ void __launch_bounds__(kDecThreads, 2) decode_fused_kernel(DecodePlan p, FusedParams f) {
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const int H = p.H;
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  __shared__ int s_slot;
  __shared__ __align__(16) float sq[kD], sk[kD], sv[kD], sa[kD];
  __shared__ __align__(16) float su[kD], sy[kD];
  __shared__ __align__(16) float redx[kDecThreads / 32][kD], redy[kDecThreads / 32][kD];
  __shared__ float rn[kDecThreads / 32], rkq[4], ro[4];
  __shared__ float sbeta;
  __shared__ float taps[kC3][kConvW];  // read only by the thread that wrote it

  if (tid == 0) {
    int slot = p.slot_ids[n];
    if (slot < 0 || slot >= p.n_slots) {
      raise_error(p.err, ERR_BAD_SLOT);
      slot = -1;
    } else if (!claim_state(p.claims, ((int64_t)slot * H + h) * kClaimsPerState, p.epoch)) {
      raise_error(p.err, ERR_DUP_SLOT);
      slot = -1;
    }
    s_slot = slot;
  }
  __syncthreads();
  const int slot = s_slot;
  if (slot < 0) return;

  const int64_t kStateElems = (int64_t)kD * kD;
  float *state = p.pool + ((int64_t)slot * H + h) * kStateElems;
  float4 s[kRows];
#pragma unroll
  for (int m = 0; m < kRows; ++m)
    s[m] = __ldcs(reinterpret_cast<const float4 *>(state + (w * kRows + m) * kD) + l);

  const bool has_v = tid < kD;
  const int c0 = tid, c1 = 2 * kD + tid;
  T *cpool = static_cast<T *>(f.conv_pool) + ((int64_t)slot * H + h) * kC3 * (kConvW - 1);
  const float *cw = f.conv_w + (int64_t)h * kC3 * kConvW;
#pragma unroll
  for (int i = 0; i < kConvW; ++i) {
    taps[c0][i] = cw[c0 * kConvW + i];
    if (has_v) taps[c1][i] = cw[c1 * kConvW + i];
  }
  float h0[kConvW - 1], h1[kConvW - 1];
#pragma unroll
  for (int i = 0; i < kConvW - 1; ++i) {
    h0[i] = to_f32(cpool[c0 * (kConvW - 1) + i]);
    h1[i] = has_v ? to_f32(cpool[c1 * (kConvW - 1) + i]) : 0.f;
  }
  const T *g = (const T *)p.g, *beta = (const T *)p.beta, *gate = (const T *)f.gate;
  T *out = (T *)p.out;
  const float nw = has_v ? f.norm_w[tid] : 0.f;
  const float qscale = rsqrtf((float)kD);

  for (int j = 0; j < p.n_tok; ++j) {
    const int64_t t = (int64_t)n * p.n_tok + j, row = t * H + h;
    const float x0 = raw_input<T>(f, t, H, h, kD, kD, c0);
    const float x1 = has_v ? raw_input<T>(f, t, H, h, kD, kD, c1) : 0.f;
    const float gr = has_v ? to_f32(g[row * kD + tid]) : 0.f;
    const float gt = has_v ? to_f32(gate[row * kD + tid]) : 0.f;
    if (tid == 0) sbeta = to_f32(beta[row]);
    float y0 = taps[c0][kConvW - 1] * x0, y1 = has_v ? taps[c1][kConvW - 1] * x1 : 0.f;
#pragma unroll
    for (int i = 0; i < kConvW - 1; ++i) {
      y0 = fmaf(taps[c0][i], h0[i], y0);
      if (has_v) y1 = fmaf(taps[c1][i], h1[i], y1);
    }
#pragma unroll
    for (int i = 0; i + 1 < kConvW - 1; ++i) { h0[i] = h0[i + 1]; h1[i] = h1[i + 1]; }
    h0[kConvW - 2] = x0;
    h1[kConvW - 2] = x1;
    y0 = act_f(y0, f.act);
    y1 = act_f(y1, f.act);
    float ysq = y0 * y0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ysq += __shfl_xor_sync(0xffffffffu, ysq, off);
    if (l == 0) rn[w] = ysq;  // warps 0-3: |q~|^2 partials, 4-7: |k~|^2
    __syncthreads();
    // the recurrence takes q, k, v in the call's element type (as the prefill does)
    if (has_v) {
      const float qn = (rn[0] + rn[1]) + (rn[2] + rn[3]);
      sq[tid] = to_f32(from_f32<T>(y0 * (qn > 0.f ? rsqrtf(qn) : 0.f) * qscale));
      sv[tid] = to_f32(from_f32<T>(y1));
      sa[tid] = expf(gr);
    } else {
      const float kn = (rn[4] + rn[5]) + (rn[6] + rn[7]);
      sk[tid - kD] = to_f32(from_f32<T>(y0 * (kn > 0.f ? rsqrtf(kn) : 0.f)));
    }
    __syncthreads();
    // the recurrence step of the 128 x 128 decode kernels
    if (has_v) {
      float kq = sq[tid] * sk[tid];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
      if (l == 0) rkq[w] = kq;
    }
    float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f), y4 = x4;
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
      const int i = w * kRows + m;
      const float ai = sa[i], ki = sk[i], qi = sq[i];
      s[m].x *= ai; s[m].y *= ai; s[m].z *= ai; s[m].w *= ai;
      x4.x = fmaf(ki, s[m].x, x4.x); x4.y = fmaf(ki, s[m].y, x4.y);
      x4.z = fmaf(ki, s[m].z, x4.z); x4.w = fmaf(ki, s[m].w, x4.w);
      y4.x = fmaf(qi, s[m].x, y4.x); y4.y = fmaf(qi, s[m].y, y4.y);
      y4.z = fmaf(qi, s[m].z, y4.z); y4.w = fmaf(qi, s[m].w, y4.w);
    }
    *reinterpret_cast<float4 *>(&redx[w][4 * l]) = x4;
    *reinterpret_cast<float4 *>(&redy[w][4 * l]) = y4;
    __syncthreads();
    if (has_v) {
      float xs = 0.f;
#pragma unroll
      for (int ww = 0; ww < kDecThreads / 32; ++ww) xs += redx[ww][tid];
      su[tid] = sbeta * (sv[tid] - xs);
    } else {
      float ys = 0.f;
#pragma unroll
      for (int ww = 0; ww < kDecThreads / 32; ++ww) ys += redy[ww][tid - kD];
      sy[tid - kD] = ys;
    }
    __syncthreads();
    // output o = y + u (k . q), then its RMSNorm and gate
    float o = 0.f;
    if (has_v) {
      o = fmaf(su[tid], (rkq[0] + rkq[1]) + (rkq[2] + rkq[3]), sy[tid]);
      float osq = o * o;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) osq += __shfl_xor_sync(0xffffffffu, osq, off);
      if (l == 0) ro[w] = osq;
    }
    const float4 u4 = *reinterpret_cast<const float4 *>(&su[4 * l]);
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
      const float ki = sk[w * kRows + m];
      s[m].x = fmaf(ki, u4.x, s[m].x); s[m].y = fmaf(ki, u4.y, s[m].y);
      s[m].z = fmaf(ki, u4.z, s[m].z); s[m].w = fmaf(ki, u4.w, s[m].w);
    }
    if (p.per_tok) {
      float *pt = p.per_tok + (t * H + h) * kStateElems;
#pragma unroll
      for (int m = 0; m < kRows; ++m)
        __stcs(reinterpret_cast<float4 *>(pt + (w * kRows + m) * kD) + l, s[m]);
    }
    // past this barrier only ro is still read (just below); the next token
    // writes ro four barriers later, so its staging can start at once
    __syncthreads();
    if (has_v) {
      const float r = rsqrtf(((ro[0] + ro[1]) + (ro[2] + ro[3])) / (float)kD + f.eps);
      out[row * kD + tid] = from_f32<T>(o * r * nw * sigmoid_f(gt));
    }
  }

#pragma unroll
  for (int m = 0; m < kRows; ++m)
    __stcs(reinterpret_cast<float4 *>(state + (w * kRows + m) * kD) + l, s[m]);
#pragma unroll
  for (int i = 0; i < kConvW - 1; ++i) {
    cpool[c0 * (kConvW - 1) + i] = from_f32<T>(h0[i]);
    if (has_v) cpool[c1 * (kConvW - 1) + i] = from_f32<T>(h1[i]);
  }
}

template <typename T>
void launch_rms_vec(const PrefillPlan &p, const FusedParams &f, const T *o, T *out, unsigned grid) {
  if (p.dv == 128) rms_gate_kernel<T, 4><<<grid, 256, 0, p.stream>>>(p, f, o, out);
  else if (p.dv == 64) rms_gate_kernel<T, 2><<<grid, 256, 0, p.stream>>>(p, f, o, out);
  else rms_gate_kernel<T, 1><<<grid, 256, 0, p.stream>>>(p, f, o, out);
}

}  // namespace

cudaError_t launch_conv_prefill(const PrefillPlan &p, const FusedParams &f) {
  if (p.T_total == 0) return cudaSuccess;
  const int64_t units = (p.T_total + kConvRun - 1) / kConvRun * p.H;
  const unsigned grid = (unsigned)((units + kConvUnits - 1) / kConvUnits);
  if (p.dtype == KDA_BF16)
    conv_prefill_kernel<__nv_bfloat16><<<grid, kConvThreads, 0, p.stream>>>(p, f);
  else
    conv_prefill_kernel<float><<<grid, kConvThreads, 0, p.stream>>>(p, f);
  return cudaGetLastError();
}

cudaError_t launch_conv_state(const PrefillPlan &p, const FusedParams &f) {
  if (p.B == 0) return cudaSuccess;
  const int C = 2 * p.dk + p.dv;
  dim3 grid(p.B, p.H);
  const int threads = (C + 31) / 32 * 32;
  if (p.dtype == KDA_BF16)
    conv_state_kernel<__nv_bfloat16><<<grid, threads, 0, p.stream>>>(p, f);
  else
    conv_state_kernel<float><<<grid, threads, 0, p.stream>>>(p, f);
  return cudaGetLastError();
}

cudaError_t launch_rms_gate(const PrefillPlan &p, const FusedParams &f, const void *o, void *out) {
  const int64_t rows = (int64_t)p.T_total * p.H;
  if (rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + 8 * kRmsRows - 1) / (8 * kRmsRows));
  // dv is 16, 32, 64 or 128 (checked by every entry point) and every pointer
  // is 16-byte aligned: each lane's E elements are one aligned vector
  using bf = __nv_bfloat16;
  if (p.dtype == KDA_BF16)
    launch_rms_vec<bf>(p, f, static_cast<const bf *>(o), static_cast<bf *>(out), grid);
  else
    launch_rms_vec<float>(p, f, static_cast<const float *>(o), static_cast<float *>(out), grid);
  return cudaGetLastError();
}

cudaError_t launch_decode_fused(const DecodePlan &p, const FusedParams &f) {
  if (p.N == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((int64_t)p.N * p.H);
  if (p.dtype == KDA_BF16)
    decode_fused_kernel<__nv_bfloat16><<<grid, kDecThreads, 0, p.stream>>>(p, f);
  else
    decode_fused_kernel<float><<<grid, kDecThreads, 0, p.stream>>>(p, f);
  return cudaGetLastError();
}

}  // namespace kda
