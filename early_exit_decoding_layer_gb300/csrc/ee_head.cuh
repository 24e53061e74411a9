// Vocabulary-head statistics shared by the GEMV and the tensor-core GEMM:
// online (max, sum of exp(z - max), argmax) over vocabulary rows, the merge
// of per-CTA partials, and the checkpoint decision with list compaction.
#pragma once

#include <math.h>

#include "ee_common.cuh"
#include "ee_kernels.cuh"

namespace ee {

struct Stat {
  float mx, sum;
  int arg;
};

EE_DEV void stat_push(Stat& s, float z, int idx) {
  if (z > s.mx) {
    s.sum = s.sum * expf(s.mx - z) + 1.0f;
    s.mx = z;
    s.arg = idx;
  } else {
    s.sum += expf(z - s.mx);
    if (z == s.mx && idx < s.arg) s.arg = idx;
  }
}

EE_DEV Stat stat_merge(Stat a, Stat b) {
  if (b.sum == 0.0f) return a;
  if (a.sum == 0.0f) return b;
  Stat r;
  r.mx = fmaxf(a.mx, b.mx);
  r.sum = a.sum * expf(a.mx - r.mx) + b.sum * expf(b.mx - r.mx);
  r.arg = a.mx > b.mx ? a.arg : (b.mx > a.mx ? b.arg : min(a.arg, b.arg));
  return r;
}

EE_DEV Stat stat_warp_merge(Stat s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Stat t;
    t.mx = __shfl_xor_sync(0xffffffffu, s.mx, o);
    t.sum = __shfl_xor_sync(0xffffffffu, s.sum, o);
    t.arg = __shfl_xor_sync(0xffffffffu, s.arg, o);
    s = stat_merge(s, t);
  }
  return s;
}

// Exit decision at a checkpoint (one thread): list entry m of the full list lf
// has score[m * stride]; it exits when the score is above gamma (strict).
// Rebuilds the full list (the sequences that stay, in order) and the exit
// list (the previous exit list le merged with the newly exited, by id), and
// records the scores and exit layers.
// A sequence with a forced exit layer (lists->forced[seq] >= 0) exits at
// that checkpoint whatever its score.
EE_DEV bool checkpoint_exits(const StepLists* lists, int seq, float conf, float gamma, int ckpt_layer) {
  const int f = lists->forced[seq];
  return f >= 0 ? f == ckpt_layer : conf > gamma;
}

EE_DEV void checkpoint_decide(float gamma, int ckpt_index, int ckpt_layer, const float* score, int stride,
                              const int32_t* lf, const int32_t* le, int nrows, float* conf_out, int32_t* exit_layer,
                              StepLists* lists) {
  int32_t nfull = 0, nexit = 0;
  int32_t newly[EE_MAX_BATCH];
  int nnew = 0;
  for (int m = 0; m < nrows; ++m) {
    const int seq = lf[1 + m];
    const float conf = score[m * stride];
    conf_out[seq * EE_MAX_CHECKPOINTS + ckpt_index] = conf;
    if (checkpoint_exits(lists, seq, conf, gamma, ckpt_layer)) {
      newly[nnew++] = seq;
      exit_layer[seq] = ckpt_layer;
    } else {
      lists->full[1 + nfull++] = seq;
    }
  }
  const int nold = min(le[0], EE_MAX_BATCH);
  int a = 0, b = 0;
  while (a < nold || b < nnew) {
    const bool take_old = b >= nnew || (a < nold && le[1 + a] < newly[b]);
    lists->exitl[1 + nexit++] = take_old ? le[1 + a++] : newly[b++];
  }
  lists->full[0] = nfull;
  lists->exitl[0] = nexit;
}

// Run by threads 0 .. nthreads-1 (whole warps) of the last CTA to finish a
// head launch: merges the nparts partials head_part[part][m] (max, sum,
// argmax) of the nrows sequences of list lf, then writes the head's results
// (confidence and argmax, the final token, or the checkpoint decision with
// the rebuilt full/exit lists).  res: shared scratch of 2 * EE_MAX_BATCH
// floats.  The threads meet on named barrier 1.
EE_DEV void head_finalize_group(const LinearParams& p, int nparts, const int32_t* lf, const int32_t* le, int nrows,
                                float* res, int nthreads) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;
  __threadfence();
  for (int m = warp; m < nrows; m += nwarps) {
    Stat s = {-INFINITY, 0.0f, 0x7fffffff};
    for (int c = lane; c < nparts; c += 32) {
      const float* src = p.head_part + ((size_t)c * EE_MAX_BATCH + m) * 4;
      s = stat_merge(s, Stat{__ldcg(src), __ldcg(src + 1), __float_as_int(__ldcg(src + 2))});
    }
    s = stat_warp_merge(s);
    if (lane == 0) {
      res[2 * m] = 1.0f / s.sum;  // max softmax = exp(zmax - lse) = 1 / sum exp(z - zmax)
      res[2 * m + 1] = __int_as_float(s.arg);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  if (tid == 0) {
    if (p.head_mode == HEAD_CONF_ARGMAX) {
      for (int m = 0; m < nrows; ++m) {
        p.conf_out[m] = res[2 * m];
        p.argmax_out[m] = __float_as_int(res[2 * m + 1]);
      }
    } else if (p.head_mode == HEAD_FINAL) {
      for (int m = 0; m < nrows; ++m) p.argmax_out[lf[1 + m]] = __float_as_int(res[2 * m + 1]);
    } else {  // HEAD_CHECKPOINT: decide, then rebuild the two sub-batch lists
      if (p.argmax_out) {  // exit-head tokens: an exiting sequence emits this head's argmax
        const float gamma = p.gamma[p.ckpt_index];
        for (int m = 0; m < nrows; ++m)
          if (checkpoint_exits(p.lists, lf[1 + m], res[2 * m], gamma, p.ckpt_layer))
            p.argmax_out[lf[1 + m]] = __float_as_int(res[2 * m + 1]);
      }
      checkpoint_decide(p.gamma[p.ckpt_index], p.ckpt_index, p.ckpt_layer, res, 2, lf, le, nrows, p.conf_out,
                        p.exit_layer, p.lists);
    }
    __threadfence();
    *p.head_counter = 0;
  }
}

EE_DEV void head_finalize(const LinearParams& p, int nparts, const int32_t* lf, const int32_t* le, int nrows,
                          float* res) {
  head_finalize_group(p, nparts, lf, le, nrows, res, (int)blockDim.x);
}

}  // namespace ee
