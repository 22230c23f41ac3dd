// Schedule IR: geometry planning, lowering, validation, serialisation.
// See schedule.hpp for the model and the serialised format.
#include "schedule.hpp"

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <numeric>

namespace amk {

namespace {

int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

int elt_bits(int fmt) { return fmt == AMK_FORMAT_BF16 ? 16 : fmt == AMK_FORMAT_INT8 ? 8 : 4; }

int ilog2(int v) {
  int r = 0;
  while ((1 << r) < v) ++r;
  return r;
}

bool plan_matrix(int fmt, int rows, int K, MatGeom* m, std::string* why, const char* name) {
  m->fmt = fmt;
  m->rows = rows;
  m->K = K;
  if (fmt == AMK_FORMAT_INT4 && K % 128) {
    *why = std::string(name) + ": int4 needs in_features % 128 == 0";
    return false;
  }
  // Kt: tile width.  A consumer thread owns one 8-element chunk of every
  // K tile, so it keeps 8 * nkt activation floats in registers.
  int best_kt = 0;
  int64_t best_kp = 0;
  for (int kt : {2048, 1024, 512, 256}) {
    int64_t kp = round_up(K, kt);
    if (kp / kt * 8 > kMaxHReg) continue;
    if (best_kt == 0 || kp < best_kp) {
      best_kt = kt;
      best_kp = kp;
    }
  }
  if (!best_kt) {
    *why = std::string(name) + ": in_features too large for register-resident activations";
    return false;
  }
  m->Kt = best_kt;
  m->Kp = (int32_t)best_kp;
  m->nkt = (int32_t)(best_kp / best_kt);
  const int64_t tile_elems = (int64_t)kStageBytes * 8 / elt_bits(fmt);
  m->Rt = (int32_t)(tile_elems / best_kt);
  m->rows_padded = (int32_t)round_up(rows, m->Rt);
  m->cpr_shift = ilog2(best_kt / 8);
  m->tile_bytes = kStageBytes;
  m->side_bytes = 0;
  if (fmt == AMK_FORMAT_INT4) {
    // per tile: Rt rows x (Kt/128) groups of (fp16 scale, u8 zero)
    m->side_bytes = round_up((int64_t)m->Rt * (best_kt / 128) * 3, 16);
    if (m->side_bytes > kSideBytes) {
      *why = std::string(name) + ": int4 side data exceeds a stage";
      return false;
    }
  }
  m->rb_bytes = (int64_t)m->nkt * (m->tile_bytes + m->side_bytes);
  m->bytes = (int64_t)m->n_rb() * m->rb_bytes;
  return true;
}

}  // namespace

amk_status plan_geometry(const amk_config& c, const BuildOptions& opt, ModelGeom* g,
                         std::string* why) {
  if (c.n_layers <= 0 || c.hidden <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 ||
      c.head_dim <= 0 || c.ffn <= 0 || c.vocab <= 0 || c.max_seq <= 0 ||
      !(c.rms_eps >= 0.0f) || !(c.rope_theta > 0.0f)) {
    *why = "config has a non-positive size";
    return AMK_ERR_INVALID_ARG;
  }
  for (int f : {c.weight_format, c.lm_head_format})
    if (f < AMK_FORMAT_BF16 || f > AMK_FORMAT_INT4) {
      *why = "unknown weight format";
      return AMK_ERR_INVALID_ARG;
    }
  if (c.head_dim != 64 && c.head_dim != 128) {
    *why = "head_dim must be 64 or 128";
    return AMK_ERR_UNSUPPORTED;
  }
  if (c.n_heads % c.n_kv_heads) {
    *why = "n_heads must be a multiple of n_kv_heads";
    return AMK_ERR_UNSUPPORTED;
  }
  const int group = c.n_heads / c.n_kv_heads;
  if (group * c.head_dim > kMaxGroupDim) {
    *why = "(n_heads / n_kv_heads) * head_dim must be <= 512";
    return AMK_ERR_UNSUPPORTED;
  }
  if (c.hidden % 8 || c.ffn % 8) {
    *why = "hidden and ffn must be multiples of 8";
    return AMK_ERR_UNSUPPORTED;
  }
  if (opt.num_ctas <= 0 || opt.num_ctas > 4096) {
    *why = "num_ctas must be in [1, 4096]";
    return AMK_ERR_INVALID_ARG;
  }
  g->cfg = c;
  const int qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
  const int lm_fmt = c.tied_embeddings ? AMK_FORMAT_BF16 : c.lm_head_format;
  if (!plan_matrix(c.weight_format, qd + 2 * kvd, c.hidden, &g->mat[M_QKV], why, "qkv") ||
      !plan_matrix(c.weight_format, c.hidden, qd, &g->mat[M_O], why, "o_proj") ||
      !plan_matrix(c.weight_format, 2 * c.ffn, c.hidden, &g->mat[M_GU], why, "gate_up") ||
      !plan_matrix(c.weight_format, c.hidden, c.ffn, &g->mat[M_DOWN], why, "down") ||
      !plan_matrix(lm_fmt, c.vocab, c.hidden, &g->mat[M_LM], why, "lm_head"))
    return AMK_ERR_UNSUPPORTED;
  g->num_ctas = opt.num_ctas;
  int splits = opt.attn_splits > 0 ? opt.attn_splits : std::max(1, opt.num_ctas / c.n_kv_heads);
  if (opt.attn_splits <= 0) splits = std::min<int>(splits, std::max(1, (c.max_seq + 15) / 16));
  if (splits > 1024) {
    *why = "attn_splits must be <= 1024";
    return AMK_ERR_INVALID_ARG;
  }
  g->splits = splits;
  g->group = group;
  g->rows_max = opt.max_rows_per_task > 0 ? std::min(opt.max_rows_per_task, kRowsMax) : kRowsMax;
  g->part_stride = group * (c.head_dim + 2);
  return AMK_OK;
}

// ------------------------------------------------------------------ builder

namespace {

struct Builder {
  const ModelGeom& g;
  Schedule s;
  std::vector<int64_t> cum_bytes;  // bytes streamed per CTA so far (load balance)
  int C;

  explicit Builder(const ModelGeom& geom) : g(geom), C(geom.num_ctas) {
    cum_bytes.assign(C, 0);
    s.queues.assign(C, {});
  }

  int counter() {
    s.counters.push_back({});
    return (int)s.counters.size() - 1;
  }

  int task(int type, int layer, int queue) {
    Task t;
    t.type = type;
    t.layer = layer;
    t.queue = queue;
    s.tasks.push_back(t);
    int id = (int)s.tasks.size() - 1;
    if (queue >= 0) s.queues[queue].push_back(id);
    return id;
  }

  void signal(int t, int c) {
    s.tasks[t].signal = c;
    s.counters[c].producers++;
  }

  void acc(int t, int buf, int64_t lo, int64_t hi, bool write) {
    if (hi > lo) s.tasks[t].acc.push_back({buf, lo, hi, write ? 1 : 0});
  }

  // Row blocks of one matrix split over the CTAs; extra blocks go to the
  // CTAs that have streamed the fewest bytes so far, so every CTA streams
  // about the same total over the whole step.  Returns the task ids.
  std::vector<int> distribute(int kind, int type, int layer) {
    const MatGeom& m = g.mat[kind];
    const int n = m.n_rb();
    std::vector<int> cnt(C, n / C);
    const int rem = n % C;
    if (rem) {
      std::vector<int> order(C);
      std::iota(order.begin(), order.end(), 0);
      std::stable_sort(order.begin(), order.end(),
                       [&](int a, int b) { return cum_bytes[a] < cum_bytes[b]; });
      for (int i = 0; i < rem; ++i) cnt[order[i]]++;
    }
    std::vector<int> ids;
    const int rb_max = std::max(1, g.rows_max / m.Rt);
    int start = 0;
    for (int c = 0; c < C; ++c) {
      if (!cnt[c]) continue;
      const int nt = (cnt[c] + rb_max - 1) / rb_max;
      int rb = start;
      for (int i = 0; i < nt; ++i) {
        const int take = cnt[c] / nt + (i < cnt[c] % nt ? 1 : 0);
        int t = task(type, layer, c);
        s.tasks[t].a[0] = rb;
        s.tasks[t].a[1] = rb + take;
        ids.push_back(t);
        rb += take;
      }
      start += cnt[c];
      cum_bytes[c] += (int64_t)cnt[c] * m.rb_bytes;
    }
    return ids;
  }

  // packed QKV rows [p0, p1) -> the ranges of Q / KVCUR they write
  void qkv_writes(int t, int layer, int64_t p0, int64_t p1) {
    const amk_config& c = g.cfg;
    const int hd = c.head_dim, half = hd / 2;
    const int64_t qd = (int64_t)c.n_heads * hd, kvd = (int64_t)c.n_kv_heads * hd;
    auto rope_region = [&](int64_t r0, int64_t r1, int64_t base, int buf, int64_t off) {
      // r0, r1 relative to the region start; pairs (2i, 2i+1) -> dims i, i + half
      for (int64_t h0 = r0 / hd * hd; h0 < r1; h0 += hd) {
        int64_t a = std::max(r0, h0) - h0, b = std::min(r1, h0 + hd) - h0;
        if (b <= a) continue;
        int64_t i0 = a / 2, i1 = (b + 1) / 2;
        acc(t, buf, off + base + h0 + i0, off + base + h0 + i1, true);
        acc(t, buf, off + base + h0 + half + i0, off + base + h0 + half + i1, true);
      }
    };
    if (p0 < qd) rope_region(p0, std::min(p1, qd), 0, B_Q, 0);
    if (p1 > qd && p0 < qd + kvd)
      rope_region(std::max(p0, qd) - qd, std::min(p1, qd + kvd) - qd, 0, B_KVCUR,
                  (int64_t)(layer * 2 + 0) * kvd);
    if (p1 > qd + kvd)
      acc(t, B_KVCUR, (int64_t)(layer * 2 + 1) * kvd + std::max(p0, qd + kvd) - qd - kvd,
          (int64_t)(layer * 2 + 1) * kvd + std::min<int64_t>(p1, qd + 2 * kvd) - qd - kvd, true);
  }

  Schedule build() {
    const amk_config& c = g.cfg;
    const int L = c.n_layers, H = c.hidden, F = c.ffn, hd = c.head_dim;
    const int64_t qd = (int64_t)c.n_heads * hd, kvd = (int64_t)c.n_kv_heads * hd;
    const int S = g.splits, G = g.group, ps = g.part_stride;

    s.buffers.resize(B_NUM);
    s.buffers[B_X] = {H, BUF_SCRATCH};
    s.buffers[B_Q] = {qd, BUF_SCRATCH};
    s.buffers[B_KVCUR] = {(int64_t)L * 2 * kvd, BUF_STATE};
    s.buffers[B_PART] = {(int64_t)c.n_kv_heads * S * ps, BUF_SCRATCH};
    s.buffers[B_O] = {qd, BUF_SCRATCH};
    s.buffers[B_A] = {F, BUF_SCRATCH};
    s.buffers[B_LOGITS] = {c.vocab, BUF_OUTPUT};

    int prev_down = -1;
    for (int l = 0; l < L; ++l) {
      const int c_qkv = counter(), c_attn = counter(), c_o = counter(), c_gu = counter(),
                c_down = counter();
      std::vector<int> tickets(c.n_kv_heads);
      for (auto& tk : tickets) tk = counter();

      // QKV
      auto qkv = distribute(M_QKV, T_QKV, l);
      const int nq = (int)qkv.size();
      for (int i = 0; i < nq; ++i) {
        int t = qkv[i];
        if (prev_down >= 0) s.tasks[t].waits.push_back({prev_down, s.counters[prev_down].producers});
        signal(t, c_qkv);
        const MatGeom& m = g.mat[M_QKV];
        int64_t p0 = s.tasks[t].a[0] * m.Rt, p1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
        if (l > 0) {
          acc(t, B_X, 0, H, false);
        } else {
          // layer 0 also writes its share of x = embedding row
          int64_t xs0 = (int64_t)H * i / nq, xs1 = (int64_t)H * (i + 1) / nq;
          s.tasks[t].a[2] = xs0;
          s.tasks[t].a[3] = xs1;
          acc(t, B_X, xs0, xs1, true);
        }
        qkv_writes(t, l, p0, p1);
      }

      // attention: one task per (kv head, split), then the completion merge
      for (int gh = 0; gh < c.n_kv_heads; ++gh) {
        for (int j = 0; j < S; ++j) {
          int t = task(T_ATTN, l, (gh * S + j) % C);
          s.tasks[t].a[0] = gh;
          s.tasks[t].a[1] = j;
          s.tasks[t].a[2] = c_attn;
          s.tasks[t].waits.push_back({c_qkv, s.counters[c_qkv].producers});
          signal(t, tickets[gh]);
          acc(t, B_Q, (int64_t)gh * G * hd, (int64_t)(gh + 1) * G * hd, false);
          if (j == S - 1) {
            acc(t, B_KVCUR, (int64_t)(l * 2 + 0) * kvd + gh * hd, (int64_t)(l * 2 + 0) * kvd + (gh + 1) * hd, false);
            acc(t, B_KVCUR, (int64_t)(l * 2 + 1) * kvd + gh * hd, (int64_t)(l * 2 + 1) * kvd + (gh + 1) * hd, false);
          }
          acc(t, B_PART, (int64_t)(gh * S + j) * ps, (int64_t)(gh * S + j + 1) * ps, true);
        }
        int cb = task(T_COMBINE, l, -1);
        s.tasks[cb].a[0] = gh;
        s.counters[tickets[gh]].completion = cb;
        signal(cb, c_attn);
        acc(cb, B_PART, (int64_t)gh * S * ps, (int64_t)(gh + 1) * S * ps, false);
        acc(cb, B_O, (int64_t)gh * G * hd, (int64_t)(gh + 1) * G * hd, true);
      }

      // O projection + residual
      for (int t : distribute(M_O, T_OPROJ, l)) {
        s.tasks[t].waits.push_back({c_attn, s.counters[c_attn].producers});
        signal(t, c_o);
        const MatGeom& m = g.mat[M_O];
        int64_t r0 = s.tasks[t].a[0] * m.Rt, r1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
        acc(t, B_O, 0, qd, false);
        acc(t, B_X, r0, r1, false);
        acc(t, B_X, r0, r1, true);
      }
      // gate/up + SwiGLU
      for (int t : distribute(M_GU, T_GATEUP, l)) {
        s.tasks[t].waits.push_back({c_o, s.counters[c_o].producers});
        signal(t, c_gu);
        const MatGeom& m = g.mat[M_GU];
        int64_t p0 = s.tasks[t].a[0] * m.Rt, p1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
        acc(t, B_X, 0, H, false);
        acc(t, B_A, p0 / 2, (p1 + 1) / 2, true);
      }
      // down + residual
      for (int t : distribute(M_DOWN, T_DOWN, l)) {
        s.tasks[t].waits.push_back({c_gu, s.counters[c_gu].producers});
        signal(t, c_down);
        const MatGeom& m = g.mat[M_DOWN];
        int64_t r0 = s.tasks[t].a[0] * m.Rt, r1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
        acc(t, B_A, 0, F, false);
        acc(t, B_X, r0, r1, false);
        acc(t, B_X, r0, r1, true);
      }
      prev_down = c_down;
    }

    s.body_len.resize(C);
    for (int q = 0; q < C; ++q) s.body_len[q] = (int)s.queues[q].size();

    // LM head (skipped by prefill)
    for (int t : distribute(M_LM, T_LMHEAD, L - 1)) {
      s.tasks[t].waits.push_back({prev_down, s.counters[prev_down].producers});
      const MatGeom& m = g.mat[M_LM];
      int64_t r0 = s.tasks[t].a[0] * m.Rt, r1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
      acc(t, B_X, 0, H, false);
      acc(t, B_LOGITS, r0, r1, true);
    }
    return std::move(s);
  }
};

}  // namespace

Schedule build_schedule(const ModelGeom& g) { return Builder(g).build(); }

// ---------------------------------------------------------------- validator

namespace {

std::string fmt_msg(const char* f, long long a = 0, long long b = 0, long long c = 0) {
  char buf[256];
  snprintf(buf, sizeof buf, f, a, b, c);
  return buf;
}

Report fail(std::string m) {
  Report r;
  r.ok = false;
  r.msg = std::move(m);
  return r;
}

}  // namespace

Report validate(const Schedule& s) {
  const int64_t T = (int64_t)s.tasks.size(), NC = (int64_t)s.counters.size(),
                NQ = (int64_t)s.queues.size(), NB = (int64_t)s.buffers.size();
  if ((int64_t)s.body_len.size() != NQ) return fail("body_len size differs from queue count");

  // ---- referential integrity ------------------------------------------
  std::vector<int32_t> producers(NC, 0);
  std::vector<std::vector<int32_t>> prod_list(NC);
  for (int64_t t = 0; t < T; ++t) {
    const Task& k = s.tasks[t];
    if (k.type < 0 || k.type >= T_NUM_TYPES) return fail(fmt_msg("task %lld: bad type", t));
    if (k.queue < -1 || k.queue >= NQ) return fail(fmt_msg("task %lld: bad queue %lld", t, k.queue));
    for (const Wait& w : k.waits)
      if (w.counter < 0 || w.counter >= NC) return fail(fmt_msg("task %lld: wait on bad counter", t));
    if (k.signal < -1 || k.signal >= NC) return fail(fmt_msg("task %lld: bad signal counter", t));
    if (k.signal >= 0) {
      producers[k.signal]++;
      prod_list[k.signal].push_back((int32_t)t);
    }
    if (k.acc.empty()) return fail(fmt_msg("task %lld writes and reads nothing", t));
    bool writes = false;
    for (const Access& a : k.acc) {
      if (a.buffer < 0 || a.buffer >= NB) return fail(fmt_msg("task %lld: bad buffer", t));
      if (a.lo < 0 || a.hi <= a.lo || a.hi > s.buffers[a.buffer].size)
        return fail(fmt_msg("task %lld: access [%lld, %lld) out of its buffer", t, a.lo, a.hi));
      writes |= a.write != 0;
    }
    if (!writes) return fail(fmt_msg("task %lld writes nothing (unreachable work)", t));
  }
  std::vector<int32_t> completion_of(T, -1);
  for (int64_t c = 0; c < NC; ++c) {
    const Counter& k = s.counters[c];
    if (k.producers != producers[c])
      return fail(fmt_msg("counter %lld: declares %lld producers, %lld tasks signal it", c,
                          k.producers, producers[c]));
    if (k.completion != -1) {
      if (k.completion < 0 || k.completion >= T) return fail(fmt_msg("counter %lld: bad completion", c));
      if (s.tasks[k.completion].queue != -1)
        return fail(fmt_msg("counter %lld: completion task is queued", c));
      if (completion_of[k.completion] != -1)
        return fail(fmt_msg("task %lld completes two counters", k.completion));
      if (!s.tasks[k.completion].waits.empty())
        return fail(fmt_msg("completion task %lld waits", k.completion));
      if (k.producers == 0) return fail(fmt_msg("counter %lld: completion without producers", c));
      completion_of[k.completion] = (int32_t)c;
    }
  }
  std::vector<int32_t> lane_pos(T, 0), lane_of(T, -1);
  for (int64_t q = 0; q < NQ; ++q) {
    const auto& items = s.queues[q];
    if (s.body_len[q] < 0 || s.body_len[q] > (int)items.size())
      return fail(fmt_msg("queue %lld: bad body length", q));
    for (size_t i = 0; i < items.size(); ++i) {
      int32_t t = items[i];
      if (t < 0 || t >= T) return fail(fmt_msg("queue %lld: bad task id", q));
      if (s.tasks[t].queue != q) return fail(fmt_msg("task %lld listed in queue %lld", t, q));
      if (lane_of[t] != -1) return fail(fmt_msg("task %lld queued twice", t));
      lane_of[t] = (int32_t)q;
      lane_pos[t] = (int32_t)i + 1;
    }
  }
  int64_t n_lanes = NQ;
  for (int64_t t = 0; t < T; ++t) {
    if (s.tasks[t].queue >= 0 && lane_of[t] == -1) return fail(fmt_msg("task %lld not in its queue", t));
    if (s.tasks[t].queue == -1) {
      if (completion_of[t] == -1) return fail(fmt_msg("task %lld has no queue and completes nothing", t));
      lane_of[t] = (int32_t)n_lanes++;
      lane_pos[t] = 1;
    }
  }

  // ---- wait thresholds: 1 <= t <= #producers ---------------------------
  for (int64_t t = 0; t < T; ++t)
    for (const Wait& w : s.tasks[t].waits)
      if (w.threshold < 1 || w.threshold > producers[w.counter])
        return fail(fmt_msg("task %lld: wait threshold %lld outside [1, %lld producers]", t,
                            w.threshold, producers[w.counter]));

  // ---- body (prefill) closure: body tasks never wait on skipped work ----
  std::vector<char> in_body(T, 0);
  for (int64_t q = 0; q < NQ; ++q)
    for (int i = 0; i < s.body_len[q]; ++i) in_body[s.queues[q][i]] = 1;
  for (int64_t t = 0; t < T; ++t)
    if (s.tasks[t].queue == -1) {
      // a completion belongs to the body iff its trigger's producers do
      bool all = true, any = false;
      for (int32_t p : prod_list[completion_of[t]]) {
        all &= in_body[p] != 0;
        any |= in_body[p] != 0;
      }
      if (any && !all) return fail(fmt_msg("completion %lld mixes body and skipped producers", t));
      in_body[t] = all ? 1 : 0;
    }
  for (int64_t t = 0; t < T; ++t) {
    if (!in_body[t]) continue;
    for (const Wait& w : s.tasks[t].waits)
      for (int32_t p : prod_list[w.counter])
        if (!in_body[p]) return fail(fmt_msg("body task %lld waits on skipped task %lld", t, p));
  }

  // ---- acyclicity of queue-order + producer->consumer edges --------------
  std::vector<std::vector<int32_t>> succ(T);
  std::vector<int32_t> indeg(T, 0);
  auto edge = [&](int32_t a, int32_t b) {
    succ[a].push_back(b);
    indeg[b]++;
  };
  for (int64_t q = 0; q < NQ; ++q)
    for (size_t i = 1; i < s.queues[q].size(); ++i) edge(s.queues[q][i - 1], s.queues[q][i]);
  for (int64_t t = 0; t < T; ++t) {
    for (const Wait& w : s.tasks[t].waits)
      for (int32_t p : prod_list[w.counter]) edge(p, (int32_t)t);
    if (completion_of[t] >= 0)
      for (int32_t p : prod_list[completion_of[t]]) edge(p, (int32_t)t);
  }
  std::vector<int32_t> topo;
  topo.reserve(T);
  for (int64_t t = 0; t < T; ++t)
    if (!indeg[t]) topo.push_back((int32_t)t);
  for (size_t i = 0; i < topo.size(); ++i)
    for (int32_t b : succ[topo[i]])
      if (--indeg[b] == 0) topo.push_back(b);
  if ((int64_t)topo.size() != T) {
    for (int64_t t = 0; t < T; ++t)
      if (indeg[t]) return fail(fmt_msg("dependency cycle through task %lld", t));
  }

  // ---- deadlock: run the queues to a fixpoint (counters only grow) -------
  {
    std::vector<int64_t> val(NC, 0);
    std::vector<size_t> head(NQ, 0);
    int64_t done = 0;
    std::vector<int32_t> pending;
    auto fire = [&](int32_t t) {
      pending.push_back(t);
      while (!pending.empty()) {
        int32_t k = pending.back();
        pending.pop_back();
        ++done;
        int32_t c = s.tasks[k].signal;
        if (c >= 0 && ++val[c] == producers[c] && s.counters[c].completion >= 0)
          pending.push_back(s.counters[c].completion);
      }
    };
    bool progress = true;
    while (progress) {
      progress = false;
      for (int64_t q = 0; q < NQ; ++q) {
        while (head[q] < s.queues[q].size()) {
          int32_t t = s.queues[q][head[q]];
          bool ready = true;
          for (const Wait& w : s.tasks[t].waits) ready &= val[w.counter] >= w.threshold;
          if (!ready) break;
          ++head[q];
          fire(t);
          progress = true;
        }
      }
    }
    for (int64_t q = 0; q < NQ; ++q)
      if (head[q] < s.queues[q].size())
        return fail(fmt_msg("deadlock: queue %lld stalls at task %lld", q, s.queues[q][head[q]]));
    if (done != T) return fail("deadlock: a completion task never fires");
  }

  // ---- races: vector clocks over lanes (queues + completion tasks) --------
  {
    const int64_t W = n_lanes;
    std::vector<int32_t> vc((size_t)T * W, 0);
    std::vector<int32_t> tmp(W);
    std::vector<int32_t> prev_in_lane(T, -1);
    for (int64_t q = 0; q < NQ; ++q)
      for (size_t i = 1; i < s.queues[q].size(); ++i) prev_in_lane[s.queues[q][i]] = s.queues[q][i - 1];
    for (int32_t t : topo) {
      int32_t* v = &vc[(size_t)t * W];
      if (prev_in_lane[t] >= 0) std::memcpy(v, &vc[(size_t)prev_in_lane[t] * W], W * sizeof(int32_t));
      auto join_all = [&](const std::vector<int32_t>& ps) {
        for (int32_t p : ps) {
          const int32_t* pv = &vc[(size_t)p * W];
          for (int64_t i = 0; i < W; ++i) v[i] = std::max(v[i], pv[i]);
        }
      };
      for (const Wait& w : s.tasks[t].waits) {
        const auto& ps = prod_list[w.counter];
        if (w.threshold == (int32_t)ps.size()) {
          join_all(ps);
        } else {
          // any `threshold` of the producers may be the ones that finished:
          // only what precedes every producer is guaranteed to precede us
          std::fill(tmp.begin(), tmp.end(), INT32_MAX);
          for (int32_t p : ps) {
            const int32_t* pv = &vc[(size_t)p * W];
            for (int64_t i = 0; i < W; ++i) tmp[i] = std::min(tmp[i], pv[i]);
          }
          for (int64_t i = 0; i < W; ++i) v[i] = std::max(v[i], tmp[i]);
        }
      }
      if (completion_of[t] >= 0) join_all(prod_list[completion_of[t]]);
      v[lane_of[t]] = lane_pos[t];
    }
    auto hb = [&](int32_t a, int32_t b) { return vc[(size_t)b * W + lane_of[a]] >= lane_pos[a]; };

    struct Acc { int64_t lo, hi; int32_t task; int32_t write; };
    std::vector<std::vector<Acc>> per_buf(NB);
    for (int64_t t = 0; t < T; ++t)
      for (const Access& a : s.tasks[t].acc) per_buf[a.buffer].push_back({a.lo, a.hi, (int32_t)t, a.write});
    for (int64_t b = 0; b < NB; ++b) {
      auto& v = per_buf[b];
      std::vector<Acc> writes;
      for (auto& a : v)
        if (a.write) writes.push_back(a);
      std::sort(v.begin(), v.end(), [](const Acc& x, const Acc& y) { return x.lo < y.lo; });
      for (const Acc& w : writes) {
        // every access overlapping w: the sorted prefix with lo < w.hi
        for (const Acc& a : v) {
          if (a.lo >= w.hi) break;
          if (a.hi <= w.lo || a.task == w.task) continue;
          if (!hb(w.task, a.task) && !hb(a.task, w.task))
            return fail(fmt_msg("race on buffer %lld between tasks %lld and %lld", b, w.task, a.task));
        }
      }
    }
  }

  // ---- outputs: every element of an output buffer is written ------------
  for (int64_t b = 0; b < NB; ++b) {
    if (s.buffers[b].kind != BUF_OUTPUT) continue;
    std::vector<std::pair<int64_t, int64_t>> iv;
    for (const Task& k : s.tasks)
      for (const Access& a : k.acc)
        if (a.buffer == b && a.write) iv.push_back({a.lo, a.hi});
    std::sort(iv.begin(), iv.end());
    int64_t covered = 0;
    for (auto& p : iv) {
      if (p.first > covered) break;
      covered = std::max(covered, p.second);
    }
    if (covered < s.buffers[b].size)
      return fail(fmt_msg("output buffer %lld: element %lld is never written", b, covered));
  }

  Report ok;
  ok.msg = fmt_msg("accepted: %lld tasks, %lld counters, %lld queues", T, NC, NQ);
  return ok;
}

// ------------------------------------------------------------ serialisation

std::vector<int64_t> serialize(const Schedule& s) {
  int64_t nw = 0, na = 0, ni = 0;
  for (const Task& t : s.tasks) {
    nw += (int64_t)t.waits.size();
    na += (int64_t)t.acc.size();
  }
  for (const auto& q : s.queues) ni += (int64_t)q.size();
  std::vector<int64_t> o;
  o.reserve(9 + s.buffers.size() * 2 + s.counters.size() * 2 + s.tasks.size() * 12 + nw * 2 +
            na * 4 + s.queues.size() * 3 + ni);
  o.insert(o.end(), {0x414D4B53, 1, (int64_t)s.tasks.size(), (int64_t)s.counters.size(),
                     (int64_t)s.queues.size(), (int64_t)s.buffers.size(), nw, na, ni});
  for (const Buffer& b : s.buffers) o.insert(o.end(), {b.size, b.kind});
  for (const Counter& c : s.counters) o.insert(o.end(), {c.producers, c.completion});
  int64_t wb = 0, ab = 0;
  for (const Task& t : s.tasks) {
    o.insert(o.end(), {t.type, t.layer, t.queue, wb, (int64_t)t.waits.size(), t.signal, ab,
                       (int64_t)t.acc.size(), t.a[0], t.a[1], t.a[2], t.a[3]});
    wb += (int64_t)t.waits.size();
    ab += (int64_t)t.acc.size();
  }
  for (const Task& t : s.tasks)
    for (const Wait& w : t.waits) o.insert(o.end(), {w.counter, w.threshold});
  for (const Task& t : s.tasks)
    for (const Access& a : t.acc) o.insert(o.end(), {a.buffer, a.lo, a.hi, a.write});
  int64_t ib = 0;
  for (size_t q = 0; q < s.queues.size(); ++q) {
    o.insert(o.end(), {ib, (int64_t)s.queues[q].size(), (int64_t)s.body_len[q]});
    ib += (int64_t)s.queues[q].size();
  }
  for (const auto& q : s.queues)
    for (int32_t t : q) o.push_back(t);
  return o;
}

bool deserialize(const int64_t* w, size_t n, Schedule* out, std::string* why) {
  auto bad = [&](const char* m) {
    *why = m;
    return false;
  };
  if (n < 9 || w[0] != 0x414D4B53 || w[1] != 1) return bad("not a serialised schedule");
  const int64_t nt = w[2], nc = w[3], nq = w[4], nb = w[5], nw = w[6], na = w[7], ni = w[8];
  const int64_t lim = (int64_t)1 << 31;
  for (int64_t v : {nt, nc, nq, nb, nw, na, ni})
    if (v < 0 || v >= lim) return bad("schedule header sizes out of range");
  const int64_t need = 9 + nb * 2 + nc * 2 + nt * 12 + nw * 2 + na * 4 + nq * 3 + ni;
  if ((int64_t)n != need) return bad("schedule length does not match its header");
  auto fits32 = [](int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; };
  const int64_t* p = w + 9;
  Schedule s;
  s.buffers.resize(nb);
  for (auto& b : s.buffers) {
    b.size = p[0];
    if (!fits32(p[1])) return bad("bad buffer kind");
    b.kind = (int32_t)p[1];
    p += 2;
  }
  s.counters.resize(nc);
  for (auto& c : s.counters) {
    if (!fits32(p[0]) || !fits32(p[1])) return bad("bad counter");
    c.producers = (int32_t)p[0];
    c.completion = (int32_t)p[1];
    p += 2;
  }
  const int64_t* tasks = p;
  p += nt * 12;
  const int64_t* waits = p;
  p += nw * 2;
  const int64_t* accs = p;
  p += na * 4;
  s.tasks.resize(nt);
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t* r = tasks + t * 12;
    for (int i = 0; i < 8; ++i)
      if (!fits32(r[i])) return bad("task field out of range");
    Task& k = s.tasks[t];
    k.type = (int32_t)r[0];
    k.layer = (int32_t)r[1];
    k.queue = (int32_t)r[2];
    if (r[3] < 0 || r[4] < 0 || r[3] + r[4] > nw) return bad("task wait range out of bounds");
    for (int64_t i = 0; i < r[4]; ++i) {
      const int64_t* wr = waits + (r[3] + i) * 2;
      if (!fits32(wr[0]) || !fits32(wr[1])) return bad("bad wait");
      k.waits.push_back({(int32_t)wr[0], (int32_t)wr[1]});
    }
    k.signal = (int32_t)r[5];
    if (r[6] < 0 || r[7] < 0 || r[6] + r[7] > na) return bad("task access range out of bounds");
    for (int64_t i = 0; i < r[7]; ++i) {
      const int64_t* ar = accs + (r[6] + i) * 4;
      if (!fits32(ar[0]) || !fits32(ar[3])) return bad("bad access");
      k.acc.push_back({(int32_t)ar[0], ar[1], ar[2], (int32_t)ar[3]});
    }
    for (int i = 0; i < 4; ++i) k.a[i] = r[8 + i];
  }
  const int64_t* queues = p;
  p += nq * 3;
  const int64_t* items = p;
  s.queues.resize(nq);
  s.body_len.resize(nq);
  for (int64_t q = 0; q < nq; ++q) {
    const int64_t* r = queues + q * 3;
    if (r[0] < 0 || r[1] < 0 || r[0] + r[1] > ni || !fits32(r[2])) return bad("queue range out of bounds");
    for (int64_t i = 0; i < r[1]; ++i) {
      if (!fits32(items[r[0] + i])) return bad("bad queue item");
      s.queues[q].push_back((int32_t)items[r[0] + i]);
    }
    s.body_len[q] = (int32_t)r[2];
  }
  *out = std::move(s);
  return true;
}

}  // namespace amk
