// Block-causal attention oracle: plain fp64 CPU code.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
// loads this file; only the tests, the smoke check and the CPU-baseline leg of
// the benchmark do.  It shares no code, header or table with the CUDA path.
//
// What it computes is the definition of block-causal attention written out,
// with no blocking, tiling, online softmax or reordering:
//
//   "Inference for Interpretable Text-Diffusion Models", section "Background",
//   first bullet (block-causal diffusion decoding): a token attends
//   bidirectionally to every token of its own diffusion block, causally to
//   tokens of earlier blocks, and never to later blocks.
//
//   "Inference: Fewer, smaller forwards", "Advancement 1" (multi-canvas D2F
//   scheduling) and "Advancement 13" (prefix attention): canvas i attends the
//   prompt cache, earlier canvases and itself; the mask addresses keys by
//   their absolute position ("Advancement 10"), not by their storage order.
//
// Both are the same rule once every position p is given a block index
//   blk(p) = -1               if p <  P0   (completed prefix / prompt cache)
//   blk(p) = floor((p-P0)/D)  if p >= P0   (diffusion block or canvas number)
// and a query at position i may see a key at position j iff blk(j) <= blk(i).
//
// Attention itself is softmax(scale * q.k) over the allowed keys, computed in
// two passes (max, then exp/sum/weighted sum) in IEEE double precision.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

int64_t block_of(int64_t p, int64_t P0, int64_t D) {
  if (p < P0) return -1;
  return (p - P0) / D;
}

}  // namespace

extern "C" {

// Dense mask: mask[i*Tk + j] = 1 iff the query at q_pos[i] may attend the key
// at k_pos[j] (block rule above).  Returns 0, or -1 on a bad argument.
int oracle_block_causal_mask(const int64_t* q_pos, int64_t Tq, const int64_t* k_pos,
                             int64_t Tk, int64_t P0, int64_t D, uint8_t* mask) {
  if (D < 1 || Tq < 0 || Tk < 0) return -1;
  for (int64_t i = 0; i < Tq; ++i) {
    const int64_t bi = block_of(q_pos[i], P0, D);
    for (int64_t j = 0; j < Tk; ++j) {
      mask[i * Tk + j] = block_of(k_pos[j], P0, D) <= bi ? 1 : 0;
    }
  }
  return 0;
}

// Masked softmax attention over one sequence.
//   q    [Tq, Hq, d]   keys and values k, v [Tk, Hkv, d]   (row-major fp64)
//   mask [Tq, Tk]      from oracle_block_causal_mask
//   out  [Tq, Hq, d]   lse [Tq, Hq] (natural-log sum of exp of the scaled
//                      scores, may be NULL)
// Query head h reads key/value head h / (Hq / Hkv) (contiguous GQA groups).
// A query row with no allowed key is an error (-2): the block rule always
// lets a query see itself, so this never happens on valid input.
int oracle_masked_attention(const double* q, const double* k, const double* v,
                            const uint8_t* mask, int64_t Tq, int64_t Tk, int Hq, int Hkv,
                            int d, double scale, double* out, double* lse, int nthreads) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return -1;
  const int G = Hq / Hkv;
  const int64_t rows = Tq * Hq;
  if (nthreads < 1) nthreads = 1;
  std::vector<int> status(nthreads, 0);

  auto work = [&](int tid) {
    std::vector<double> s(Tk > 0 ? Tk : 1);
    for (int64_t r = tid; r < rows; r += nthreads) {
      const int64_t i = r / Hq;
      const int h = int(r % Hq);
      const int g = h / G;
      const double* qi = q + (i * Hq + h) * d;
      // pass 1: scores of the allowed keys and their maximum
      double m = -INFINITY;
      bool any = false;
      for (int64_t j = 0; j < Tk; ++j) {
        if (!mask[i * Tk + j]) continue;
        const double* kj = k + (j * Hkv + g) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += qi[c] * kj[c];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
        any = true;
      }
      double* o = out + (i * Hq + h) * d;
      if (!any) {
        status[tid] = -2;
        for (int c = 0; c < d; ++c) o[c] = NAN;
        if (lse) lse[i * Hq + h] = NAN;
        continue;
      }
      // pass 2: exponentials, their sum, and the weighted sum of values
      double denom = 0.0;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int64_t j = 0; j < Tk; ++j) {
        if (!mask[i * Tk + j]) continue;
        const double w = std::exp(s[j] - m);
        denom += w;
        const double* vj = v + (j * Hkv + g) * d;
        for (int c = 0; c < d; ++c) o[c] += w * vj[c];
      }
      for (int c = 0; c < d; ++c) o[c] /= denom;
      if (lse) lse[i * Hq + h] = m + std::log(denom);
    }
  };

  if (nthreads == 1) {
    work(0);
  } else {
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t) pool.emplace_back(work, t);
    for (auto& th : pool) th.join();
  }
  for (int t = 0; t < nthreads; ++t)
    if (status[t]) return status[t];
  return 0;
}

}  // extern "C"
