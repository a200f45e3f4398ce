// kda_recurrent.cu -- token-by-token KDA on CUDA cores, fp32 state and math.
//
// The recurrence (gated delta rule with per-channel decay, "Kimi K3 on vLLM:
// Up to 370 Tokens/sec", section "Kimi Delta Attention: a hybrid recurrent +
// full-attention stack"):
//     S' = Diag(exp g_t) S ;  u = beta_t (v_t - S'^T k_t) ;  S = S' + k_t u^T ;
//     o_t = S^T q_t = S'^T q_t + u (k_t . q_t)
//
// Columns of S evolve independently, so each thread owns one column j of one
// (sequence, head) state and keeps its dk entries in registers for the whole
// segment: every reduction over the key channels is thread-local and the
// only shared traffic is the broadcast of q, k, exp(g) per token.  A CTA is
// one warp covering 32 columns (fewer when dv < 32); the state is read once
// and written once.  Its decode form also serves the speculative verify with
// commit (replay of the previous step's accepted tokens, one state write,
// outputs of this step's tokens).  This kernel is the exact-fp32 path (fp32 inputs, shapes
// other than dk = dv = 128) and serves decode for those shapes too.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kTile = 8;  // tokens staged in shared memory at a time

struct RecArgs {
  const void *q, *k, *v, *g, *beta;
  float *pool;
  void *out;
  float *snaps;
  const int32_t *snap_slots;  // prefill retention map, or NULL (dense snapshots)
  int64_t snaps_capacity;
  int32_t snap_interval;
  int32_t H, dv, n_slots;
  // prefill: per-sequence plan; decode: slot ids (tok0 = n * n_tok)
  const SeqMeta *meta;
  const int32_t *order;
  const int32_t *slot_ids;
  int32_t n_tok;
  // decode with commit of a previous verify step (see DecodePlan)
  int32_t spec, n_prev;
  const void *k_prev, *v_prev, *g_prev, *beta_prev;
  const int32_t *accepted;
  uint32_t *err;
  uint32_t *claims;
  uint32_t epoch;
  // prefill recomputation of the units the chunked kernel handed over:
  // rerun[rank * H + h] == epoch selects a unit, every other CTA returns
  const uint32_t *rerun;
};

// R lanes share one column (R = 2 for dk = 128 keeps the column in 64
// registers per lane); lane (c, r) holds rows i = R*ii + r of column c.
template <typename Tin, int DK, int R, bool DECODE>
__global__ void __launch_bounds__(32) recurrent_kernel(RecArgs a) {
  constexpr int DKR = DK / R;
  const int lane = threadIdx.x;
  const int ncol = blockDim.x / R;
  const int c = lane / R, r = lane % R;
  const int h = blockIdx.y;
  const int j = blockIdx.z * ncol + c;
  const int H = a.H, dv = a.dv;
  const unsigned mask = 0xffffffffu >> (32 - blockDim.x);

  int64_t tok0, len, snap_off;
  int src, dst, n_acc = 0;
  if (DECODE) {
    const int n = blockIdx.x;
    const int slot = a.slot_ids[n];
    int ok = 1;
    if (slot < 0 || slot >= a.n_slots) {
      ok = 0;
      if (lane == 0) raise_error(a.err, ERR_BAD_SLOT);
    } else if (lane == 0) {
      const int64_t idx = ((int64_t)slot * H + h) * kClaimsPerState + blockIdx.z;
      if (!claim_state(a.claims, idx, a.epoch)) {
        raise_error(a.err, ERR_DUP_SLOT);
        ok = 0;
      }
    }
    ok = __shfl_sync(mask, ok, 0);
    if (ok && a.spec && a.n_prev > 0) {
      n_acc = a.accepted[n];
      if (n_acc < 0 || n_acc > a.n_prev) {  // the sequence is skipped: nothing written
        ok = 0;
        if (lane == 0) raise_error(a.err, ERR_BAD_ACCEPT);
      }
    }
    if (!ok) return;
    tok0 = (int64_t)n * a.n_tok;
    len = a.n_tok;
    src = dst = slot;
    snap_off = (int64_t)n * a.n_tok;
  } else {
    if (a.rerun && a.rerun[(int64_t)blockIdx.x * H + h] != a.epoch) return;
    const SeqMeta m = a.meta[a.order[blockIdx.x]];
    if (!m.ok) return;
    tok0 = m.tok0;
    len = m.len;
    src = m.src;
    dst = m.dst;
    snap_off = m.snap_off;
  }

  const int64_t state_elems = (int64_t)DK * dv;
  float S[DKR];
  if (src >= 0) {
    const float *s0 = a.pool + ((int64_t)src * H + h) * state_elems + (int64_t)r * dv + j;
#pragma unroll
    for (int ii = 0; ii < DKR; ++ii) S[ii] = s0[(int64_t)ii * R * dv];
  } else {
#pragma unroll
    for (int ii = 0; ii < DKR; ++ii) S[ii] = 0.f;
  }

  __shared__ float sk[kTile][DK], sq[kTile][DK], sa[kTile][DK];
  __shared__ float sv[kTile][32], sb[kTile], skq[kTile];

  const int nthr = blockDim.x;
  // Tokens [tok0, tok0 + len) of the given arrays applied to S; outputs are
  // written when q is given (a replayed token has none), snapshots when asked.
  auto run_tokens = [&](const Tin *q, const Tin *k, const Tin *v, const Tin *g, const Tin *beta,
                        Tin *out, int64_t tok0, int64_t len, bool snap) {
    for (int64_t t0 = 0; t0 < len; t0 += kTile) {
      const int nt = (int)((len - t0) < kTile ? (len - t0) : kTile);
      __syncwarp(mask);
      for (int tt = 0; tt < nt; ++tt) {
        const int64_t row = (tok0 + t0 + tt) * H + h;
        float kq = 0.f;
        for (int i = lane; i < DK; i += nthr) {
          const float kk = to_f32(k[row * DK + i]);
          const float qq = q ? to_f32(q[row * DK + i]) : 0.f;
          sk[tt][i] = kk;
          sq[tt][i] = qq;
          sa[tt][i] = expf(to_f32(g[row * DK + i]));
          kq = fmaf(kk, qq, kq);
        }
        for (int off = nthr / 2; off > 0; off >>= 1) kq += __shfl_xor_sync(mask, kq, off, nthr);
        if (r == 0) sv[tt][c] = to_f32(v[row * dv + j]);
        if (lane == 0) {
          sb[tt] = to_f32(beta[row]);
          skq[tt] = kq;
        }
      }
      __syncwarp(mask);
      for (int tt = 0; tt < nt; ++tt) {
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int ii = 0; ii < DKR; ++ii) {
          const int i = ii * R + r;
          const float s = S[ii] * sa[tt][i];
          S[ii] = s;
          x = fmaf(sk[tt][i], s, x);
          y = fmaf(sq[tt][i], s, y);
        }
#pragma unroll
        for (int off = 1; off < R; off <<= 1) {
          x += __shfl_xor_sync(mask, x, off);
          y += __shfl_xor_sync(mask, y, off);
        }
        const float u = sb[tt] * (sv[tt][c] - x);
#pragma unroll
        for (int ii = 0; ii < DKR; ++ii) S[ii] = fmaf(sk[tt][ii * R + r], u, S[ii]);
        const int64_t t = tok0 + t0 + tt;
        if (out && r == 0) out[(t * H + h) * dv + j] = from_f32<Tin>(fmaf(u, skq[tt], y));
        const int64_t done = t0 + tt + 1;
        if (snap && (a.snaps || a.snap_slots) && a.snap_interval > 0 &&
            done % a.snap_interval == 0) {
          const int64_t s = snap_off + done / a.snap_interval - 1;
          if (s < a.snaps_capacity) {
            float *base = snapshot_base(a.snaps, a.snap_slots, a.pool, s, H, h, state_elems);
            if (base) {
              float *d = base + (int64_t)r * dv + j;
#pragma unroll
              for (int ii = 0; ii < DKR; ++ii) d[(int64_t)ii * R * dv] = S[ii];
            }
          } else if (lane == 0) {
            raise_error(a.err, ERR_SNAP_CAPACITY);
          }
        }
      }
    }
  };
  auto store_state = [&](int slot) {
    float *sd = a.pool + ((int64_t)slot * H + h) * state_elems + (int64_t)r * dv + j;
#pragma unroll
    for (int ii = 0; ii < DKR; ++ii) sd[(int64_t)ii * R * dv] = S[ii];
  };

  if (DECODE && a.spec) {
    // commit the accepted tokens of the previous verify step (one write),
    // then this step's tokens for their outputs only
    run_tokens(nullptr, (const Tin *)a.k_prev, (const Tin *)a.v_prev, (const Tin *)a.g_prev,
               (const Tin *)a.beta_prev, nullptr, (int64_t)blockIdx.x * a.n_prev, n_acc, false);
    if (n_acc > 0) store_state(dst);
    run_tokens((const Tin *)a.q, (const Tin *)a.k, (const Tin *)a.v, (const Tin *)a.g,
               (const Tin *)a.beta, (Tin *)a.out, tok0, len, false);
    return;
  }
  run_tokens((const Tin *)a.q, (const Tin *)a.k, (const Tin *)a.v, (const Tin *)a.g,
             (const Tin *)a.beta, (Tin *)a.out, tok0, len, true);
  store_state(dst);
}

template <bool DECODE>
cudaError_t launch(const RecArgs &a, int dk, int dv, int nseq, int dtype, cudaStream_t st) {
  if (nseq == 0) return cudaSuccess;
  const int R = dk == 128 ? 2 : 1;
  const int ncol = (dv < 32 / R) ? dv : 32 / R;
  // decode claims one word per (slot, head, column block); dk = dv = 128 (8
  // blocks) always takes the 128 x 128 decode kernel instead
  if (DECODE && dv / ncol > kClaimsPerState) return cudaErrorInvalidConfiguration;
  dim3 grid(nseq, a.H, dv / ncol), block(ncol * R);
#define KDA_REC_CASE(DK, RR)                                                         \
  case DK:                                                                           \
    if (dtype == KDA_BF16)                                                           \
      recurrent_kernel<__nv_bfloat16, DK, RR, DECODE><<<grid, block, 0, st>>>(a);    \
    else                                                                             \
      recurrent_kernel<float, DK, RR, DECODE><<<grid, block, 0, st>>>(a);            \
    break;
  switch (dk) {
    KDA_REC_CASE(16, 1)
    KDA_REC_CASE(32, 1)
    KDA_REC_CASE(64, 1)
    KDA_REC_CASE(128, 2)
    default:
      return cudaErrorInvalidValue;
  }
#undef KDA_REC_CASE
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent_prefill(const PrefillPlan &p, bool rerun_only) {
  RecArgs a = {};
  a.rerun = rerun_only ? p.rerun : nullptr;
  a.q = p.q; a.k = p.k; a.v = p.v; a.g = p.g; a.beta = p.beta;
  a.pool = p.pool; a.out = p.out; a.snaps = p.snaps; a.snap_slots = p.snap_slots;
  a.snaps_capacity = p.snaps_capacity;
  a.snap_interval = p.snap_interval; a.H = p.H; a.dv = p.dv; a.n_slots = p.n_slots;
  a.meta = p.meta; a.order = p.order; a.err = p.err; a.claims = p.claims; a.epoch = p.epoch;
  return launch<false>(a, p.dk, p.dv, p.B, p.dtype, p.stream);
}

cudaError_t launch_recurrent_decode(const DecodePlan &p) {
  RecArgs a = {};
  a.q = p.q; a.k = p.k; a.v = p.v; a.g = p.g; a.beta = p.beta;
  a.pool = p.pool; a.out = p.out; a.snaps = p.per_tok;
  a.snaps_capacity = (int64_t)p.N * p.n_tok;
  a.snap_interval = p.per_tok ? 1 : 0;
  a.H = p.H; a.dv = p.dv; a.n_slots = p.n_slots;
  a.slot_ids = p.slot_ids; a.n_tok = p.n_tok;
  a.spec = p.spec; a.n_prev = p.n_prev; a.accepted = p.accepted;
  a.k_prev = p.k_prev; a.v_prev = p.v_prev; a.g_prev = p.g_prev; a.beta_prev = p.beta_prev;
  a.err = p.err; a.claims = p.claims; a.epoch = p.epoch;
  return launch<true>(a, p.dk, p.dv, p.N, p.dtype, p.stream);
}

}  // namespace kda
