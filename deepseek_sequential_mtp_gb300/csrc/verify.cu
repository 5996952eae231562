// spec_verify: exact speculative verification of gamma drafts per request.
//
// Semantics: "M7.6 - DeepSeek MTP: Sequential Modules, Teacher Forcing, and
// Speculative Runtime" §0x09 (accept with min(1, p/q), correct from the
// normalised positive residual, bonus from the next target row, EOS/budget
// truncation) generalised to gamma drafts by the left-to-right rule of the
// speculative-decoding page.  Uniforms: Philox4x32-10 (Salmon et al., SC'11).
//
// Layout on the GPU: one CTA of 512 threads per request.
//   phase A  warp 0: lane j evaluates draft position j (two scalar loads, one
//            Philox block, one fp64 division); a ballot picks the first
//            position that ends the round.
//   phase B  all 16 warps: stream the one row pair (or the bonus row) the
//            round samples from in 1024-element chunks with coalesced
//            16-byte loads, forming residuals in fp32 and compensated
//            (hi, lo) fp32 chunk sums.
//   phase C  warp 0: fp64 prefix over chunk sums picks the chunk holding
//            u' * mass, then rescans that one chunk (L2-resident) in index
//            order to find the smallest index whose running sum exceeds it.
// The kernel is HBM-bound: it reads 2*V*4 bytes for a rejection, V*4 for a
// bonus, plus 8*gamma bytes of scalars.
#include "common.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 1024;       // elements per chunk
constexpr int kMaxChunks = 512;    // V <= 524288
constexpr int kMaxGamma = 31;

enum Event { EV_CONTINUE = 0, EV_STOP = 1, EV_REJECT = 2, EV_INVALID_DRAFT = 3, EV_INVALID_PROBS = 4 };

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ double uniform24(uint32_t w) {
  return static_cast<double>(w >> 8) * (1.0 / 16777216.0);
}

__device__ __forceinline__ bool prob_ok(float v) { return isfinite(v) && v >= 0.0f; }

// weight of element v: residual max(p - q, 0) when q != nullptr, else p.
__device__ __forceinline__ float weight_of(float pv, float qv, bool residual) {
  return residual ? fmaxf(pv - qv, 0.0f) : pv;
}

// Error-free transformation: s + e == a + b exactly, s = fl(a + b).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
// Add x to the unevaluated sum hi + lo.
__device__ __forceinline__ void acc_add(float& hi, float& lo, float x) {
  float s, e;
  two_sum(hi, x, s, e);
  hi = s;
  lo += e;
}
__device__ __forceinline__ double chunk_value(float2 v) { return (double)v.x + (double)v.y; }

template <bool kVec4>
__global__ void __launch_bounds__(kThreads, 1)
spec_verify_kernel(int gamma, int V, const float* __restrict__ p, const float* __restrict__ q,
                   const int32_t* __restrict__ draft, uint2 key, uint32_t off_lo, uint32_t off_hi,
                   const int32_t* __restrict__ eos, const int32_t* __restrict__ remaining,
                   int32_t* __restrict__ accepted, int32_t* __restrict__ next_token,
                   int32_t* __restrict__ n_emit, int32_t* __restrict__ status) {
  __shared__ float2 s_chunk[kMaxChunks];  // (hi, lo) pairs
  __shared__ float s_w[kChunk];
  __shared__ int s_cstar;
  __shared__ double s_before, s_target;
  __shared__ int s_jstar, s_event, s_bad;
  __shared__ double s_u;

  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int budget = remaining ? remaining[r] : gamma + 1;
  const int eos_id = eos ? eos[r] : -1;

  // ---------------- phase A: the accept prefix ----------------
  if (warp == 0) {
    int ev = EV_CONTINUE;
    const int j = lane;
    if (j < gamma) {
      const int y = draft[(size_t)r * gamma + j];
      if (y < 0 || y >= V) {
        ev = EV_INVALID_DRAFT;
      } else {
        const float pj = p[((size_t)r * (gamma + 1) + j) * V + y];
        const float qj = q[((size_t)r * gamma + j) * V + y];
        if (!(prob_ok(pj) && prob_ok(qj))) {
          ev = EV_INVALID_PROBS;
        } else if (qj <= 0.0f) {
          ev = EV_INVALID_DRAFT;
        } else {
          const uint4 w = philox4x32_10(make_uint4((uint32_t)j, (uint32_t)r, off_lo, off_hi), key);
          const double ratio = fmin(1.0, (double)pj / (double)qj);
          if (!(uniform24(w.x) < ratio)) ev = EV_REJECT;
          else if (j + 1 == budget || y == eos_id) ev = EV_STOP;
        }
      }
    }
    const unsigned ended = __ballot_sync(0xffffffffu, ev != EV_CONTINUE);
    const int jstar = ended ? __ffs(ended) - 1 : gamma;
    const int evstar = __shfl_sync(0xffffffffu, ev, jstar & 31);
    if (lane == 0) {
      s_jstar = jstar;
      s_event = (jstar == gamma) ? EV_CONTINUE : evstar;
      s_bad = 0;
      const uint4 w = philox4x32_10(make_uint4((uint32_t)jstar, (uint32_t)r, off_lo, off_hi), key);
      s_u = uniform24(w.y);
      if (budget < 1) {
        s_event = -1;
      }
    }
  }
  __syncthreads();
  const int jstar = s_jstar;
  const int event = s_event;

  if (event != EV_CONTINUE && event != EV_REJECT) {
    if (threadIdx.x == 0) {
      int st = MTP_VERIFY_OK, acc = jstar;
      if (event == -1) { st = MTP_VERIFY_INVALID_BUDGET; acc = 0; }
      else if (event == EV_STOP) acc = jstar + 1;
      else if (event == EV_INVALID_DRAFT) st = MTP_VERIFY_INVALID_DRAFT;
      else if (event == EV_INVALID_PROBS) st = MTP_VERIFY_INVALID_PROBS;
      accepted[r] = acc;
      next_token[r] = -1;
      n_emit[r] = acc;
      status[r] = st;
    }
    return;
  }

  // ---------------- phase B: chunk sums of the sampled weights ----------------
  // Residual elements are formed in fp32 (one rounding each, at most 2^-24 of
  // the element).  A chunk's sum is accumulated as an unevaluated pair
  // (hi, lo) of fp32 values with error-free TwoSum steps, per lane and then
  // across the warp, so the sum of the fp32 elements is kept to ~2^-45
  // relative without FP64 instructions (GB300 issues FP64 warp instructions
  // at a small fraction of the FP32 rate).
  const bool residual = (event == EV_REJECT);
  const float* prow = p + ((size_t)r * (gamma + 1) + jstar) * V;
  const float* qrow = residual ? q + ((size_t)r * gamma + jstar) * V : prow;
  const int n_chunks = (V + kChunk - 1) / kChunk;
  bool bad = false;
  for (int c = warp; c < n_chunks; c += kWarps) {
    const int base = c * kChunk;
    float hi = 0.0f, lo = 0.0f;
    if constexpr (kVec4) {
      float4 pv[8], qv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = base + 4 * (lane + 32 * i);
        pv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        qv[i] = pv[i];
        if (e < V) {
          pv[i] = __ldcs(reinterpret_cast<const float4*>(prow + e));
          if (residual) qv[i] = __ldcs(reinterpret_cast<const float4*>(qrow + e));
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        bad |= !(prob_ok(pv[i].x) && prob_ok(pv[i].y) && prob_ok(pv[i].z) && prob_ok(pv[i].w));
        if (residual)
          bad |= !(prob_ok(qv[i].x) && prob_ok(qv[i].y) && prob_ok(qv[i].z) && prob_ok(qv[i].w));
        acc_add(hi, lo, weight_of(pv[i].x, qv[i].x, residual));
        acc_add(hi, lo, weight_of(pv[i].y, qv[i].y, residual));
        acc_add(hi, lo, weight_of(pv[i].z, qv[i].z, residual));
        acc_add(hi, lo, weight_of(pv[i].w, qv[i].w, residual));
      }
    } else {
#pragma unroll 4
      for (int i = 0; i < kChunk / 32; ++i) {
        const int e = base + lane + 32 * i;
        float pv = 0.f, qv = 0.f;
        if (e < V) {
          pv = prow[e];
          if (residual) qv = qrow[e];
        }
        bad |= !prob_ok(pv) || (residual && !prob_ok(qv));
        acc_add(hi, lo, weight_of(pv, qv, residual));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ohi = __shfl_xor_sync(0xffffffffu, hi, o);
      const float olo = __shfl_xor_sync(0xffffffffu, lo, o);
      float sum, err;
      two_sum(hi, ohi, sum, err);
      hi = sum;
      lo = (lo + olo) + err;
    }
    if (lane == 0) s_chunk[c] = make_float2(hi, lo);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&s_bad, 1);
  __syncthreads();

  // ---------------- phase C: locate u' * mass ----------------
  if (warp == 0) {
    int st = MTP_VERIFY_OK;
    int cstar = -1;
    double before = 0.0, target = 0.0;
    if (s_bad) {
      st = MTP_VERIFY_INVALID_PROBS;
    } else {
      // lane l owns chunks [l*per, (l+1)*per)
      const int per = (n_chunks + 31) / 32;
      double own = 0.0;
      for (int c = lane * per; c < min(n_chunks, (lane + 1) * per); ++c) own += chunk_value(s_chunk[c]);
      const double incl = mtp::warp_inclusive_scan(own);
      const double mass = __shfl_sync(0xffffffffu, incl, 31);
      if (!(mass > 0.0)) {
        st = MTP_VERIFY_ZERO_RESIDUAL;
      } else {
        target = s_u * mass;
        // chunk holding the target (or the last chunk with mass if rounding overshoots)
        const unsigned over = __ballot_sync(0xffffffffu, incl > target);
        const unsigned has_mass = __ballot_sync(0xffffffffu, own > 0.0);
        const int src = over ? __ffs(over) - 1 : 31 - __clz(has_mass);
        if (lane == src) {
          double run = incl - own;
          int last_pos = -1;
          double before_last = run;
          for (int c = lane * per; c < min(n_chunks, (lane + 1) * per); ++c) {
            const double cv = chunk_value(s_chunk[c]);
            if (cv > 0.0) { last_pos = c; before_last = run; }
            if (over && run + cv > target) { cstar = c; before = run; break; }
            run += cv;
          }
          if (cstar < 0) { cstar = last_pos; before = before_last; }
        }
        cstar = __shfl_sync(0xffffffffu, cstar, src);
        before = __shfl_sync(0xffffffffu, before, src);
      }
    }
    if (lane == 0) {
      s_event = st;
      s_cstar = cstar;
      s_before = before;
      s_target = target;
    }
  }
  __syncthreads();
  if (s_event != MTP_VERIFY_OK) {
    if (threadIdx.x == 0) {
      accepted[r] = jstar; next_token[r] = -1; n_emit[r] = jstar; status[r] = s_event;
    }
    return;
  }
  // stage the chosen chunk's weights in shared memory (one element per thread)
  for (int i = threadIdx.x; i < kChunk; i += kThreads) {
    const int e = s_cstar * kChunk + i;
    s_w[i] = e < V ? weight_of(prow[e], residual ? qrow[e] : 0.0f, residual) : 0.0f;
  }
  __syncthreads();
  if (warp != 0) return;
  // lane l holds elements [32l, 32l+32) of the chunk, summed in index order
  double lane_sum = 0.0;
  for (int i = 0; i < 32; ++i) lane_sum += (double)s_w[32 * lane + i];
  const double target = s_target;
  const double lincl = mtp::warp_inclusive_scan(lane_sum) + s_before;
  const unsigned lover = __ballot_sync(0xffffffffu, lincl > target);
  const unsigned lpos = __ballot_sync(0xffffffffu, lane_sum > 0.0);
  if (!lover && !lpos) {  // unreachable unless the two passes disagree on an empty chunk
    if (lane == 0) {
      accepted[r] = jstar; next_token[r] = -1; n_emit[r] = jstar; status[r] = MTP_VERIFY_ZERO_RESIDUAL;
    }
    return;
  }
  const int lsrc = lover ? __ffs(lover) - 1 : 31 - __clz(lpos);
  if (lane == lsrc) {
    double run = lincl - lane_sum;
    int pick = -1, last_pos = -1;
    const int base = s_cstar * kChunk + 32 * lane;
    for (int i = 0; i < 32; ++i) {
      const float wv = s_w[32 * lane + i];
      if (wv > 0.0f) last_pos = base + i;
      run += (double)wv;
      if (lover && run > target) { pick = base + i; break; }
    }
    if (pick < 0) pick = last_pos;
    accepted[r] = jstar;
    next_token[r] = pick;
    n_emit[r] = jstar + 1;
    status[r] = MTP_VERIFY_OK;
  }
}

}  // namespace

extern "C" mtp_status spec_verify(int R, int gamma, int V, const float* p, const float* q,
                                  const int32_t* draft, uint64_t seed, uint64_t offset,
                                  const int32_t* eos, const int32_t* remaining,
                                  int32_t* accepted, int32_t* next_token, int32_t* n_emit,
                                  int32_t* status, cudaStream_t stream) {
  if (R < 0 || gamma < 0 || V <= 0) return MTP_ERR_INVALID_ARG;
  if (gamma > kMaxGamma || V > kMaxChunks * kChunk) return MTP_ERR_UNSUPPORTED;
  if (R == 0) return MTP_OK;
  if (!p || (!draft && gamma > 0) || !accepted || !next_token || !n_emit || !status) return MTP_ERR_INVALID_ARG;
  if (gamma > 0 && !q) return MTP_ERR_INVALID_ARG;
  const uint2 key = make_uint2((uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32));
  const uint32_t olo = (uint32_t)(offset & 0xFFFFFFFFu), ohi = (uint32_t)(offset >> 32);
  mtp::prof_begin(MTP_KC_SPEC_VERIFY, stream);
  const bool vec = (V % 4 == 0) && mtp::aligned16(p) && (gamma == 0 || mtp::aligned16(q));
  if (vec)
    spec_verify_kernel<true><<<R, kThreads, 0, stream>>>(gamma, V, p, q, draft, key, olo, ohi, eos,
                                                          remaining, accepted, next_token, n_emit, status);
  else
    spec_verify_kernel<false><<<R, kThreads, 0, stream>>>(gamma, V, p, q, draft, key, olo, ohi, eos,
                                                           remaining, accepted, next_token, n_emit, status);
  mtp::note_launch();
  mtp::prof_end(MTP_KC_SPEC_VERIFY, stream);
  MTP_LAUNCH_CHECK();
  return MTP_OK;
}
