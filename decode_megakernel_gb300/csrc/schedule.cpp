// Schedule IR: geometry planning, lowering, validation, serialisation.
// See schedule.hpp for the model and the serialised format.
#include "schedule.hpp"

#include <algorithm>
#include <array>
#include <map>
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
  // K tile, so it keeps 8 * nkt activation floats in registers.  int8 and
  // int4 tiles (8 or 16 rows x 2048 codes) are in tensor-core fragment order
  // with each warp owning 256 k of every tile, so they take Kt = 2048
  // whatever K is.
  int best_kt = 0;
  int64_t best_kp = 0;
  for (int kt : {2048, 1024, 512, 256}) {
    if (fmt != AMK_FORMAT_BF16 && kt != 2048) continue;
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
  if (c.n_layers > kMaxVersions) {
    *why = "n_layers must be <= 4096";
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
  g->part_stride = (group * (c.head_dim + 2) + 3) / 4 * 4;
  if (g->mat[M_QKV].Rt % 2) {
    *why = "qkv tiles must hold an even number of rows (RoPE pairs)";
    return AMK_ERR_UNSUPPORTED;
  }
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

  int task(int type, int layer, int queue) {
    Task t;
    t.type = type;
    t.layer = layer;
    t.queue = queue;
    s.tasks.push_back(t);
    int id = (int)s.tasks.size() - 1;
    s.queues[queue].push_back(id);
    return id;
  }

  void acc(int t, int buf, int64_t lo, int64_t hi, bool write, int version) {
    if (hi > lo) s.tasks[t].acc.push_back({buf, lo, hi, write ? 1 : 0, version});
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

  // Packed QKV rows [p0, p1) -> the QKV words and KV-cache row elements
  // they write.  Packed order is per KV head g: its `group` query heads,
  // then its k head (both with RoPE pairs (i, i + hd/2) in adjacent rows),
  // then its v head.
  void qkv_writes(int t, int layer, int64_t p0, int64_t p1, int v) {
    const amk_config& c = g.cfg;
    const int hd = c.head_dim, half = hd / 2, G = g.group;
    const int64_t gw = (int64_t)(G + 2) * hd, kvd = (int64_t)c.n_kv_heads * hd;
    for (int64_t h0 = p0 / hd * hd; h0 < p1; h0 += hd) {   // one head of rows at a time
      const int64_t a = std::max(p0, h0) - h0, b = std::min(p1, h0 + hd) - h0;
      if (b <= a) continue;
      const int64_t grp = h0 / gw, slot = (h0 % gw) / hd;   // slot G: k, G + 1: v
      const int64_t base = grp * gw + slot * hd;
      if (slot <= G) {
        const int64_t i0 = a / 2, i1 = (b + 1) / 2;
        acc(t, B_QKV, base + i0, base + i1, true, v);
        acc(t, B_QKV, base + half + i0, base + half + i1, true, v);
        if (slot == G) {
          const int64_t kb = (int64_t)(layer * 2 + 0) * kvd + grp * hd;
          acc(t, B_KVROW, kb + i0, kb + i1, true, 0);
          acc(t, B_KVROW, kb + half + i0, kb + half + i1, true, 0);
        }
      } else {
        acc(t, B_QKV, base + a, base + b, true, v);
        const int64_t vb = (int64_t)(layer * 2 + 1) * kvd + grp * hd;
        acc(t, B_KVROW, vb + a, vb + b, true, 0);
      }
    }
  }

  Schedule build() {
    const amk_config& c = g.cfg;
    const int L = c.n_layers, H = c.hidden, F = c.ffn, hd = c.head_dim;
    const int64_t qd = (int64_t)c.n_heads * hd, kvd = (int64_t)c.n_kv_heads * hd;
    const int S = g.splits, G = g.group, ps = g.part_stride, NKV = c.n_kv_heads;
    const int64_t gw = (int64_t)(G + 2) * hd;

    s.versions = L;
    s.buffers.resize(B_NUM);
    s.buffers[B_XRES] = {H, BUF_TAGGED};
    s.buffers[B_XMID] = {H, BUF_TAGGED};
    s.buffers[B_QKV] = {NKV * gw, BUF_TAGGED};
    s.buffers[B_PART] = {(int64_t)NKV * S * ps, BUF_TAGGED};
    s.buffers[B_O] = {qd, BUF_TAGGED};
    s.buffers[B_A] = {F, BUF_TAGGED};
    s.buffers[B_KVROW] = {(int64_t)L * 2 * kvd, BUF_STATE};
    s.buffers[B_LOGITS] = {c.vocab, BUF_OUTPUT};

    for (int l = 0; l < L; ++l) {
      const int v = l + 1;   // version written by every tagged write of layer l
      // QKV: rmsnorm(x_res) (layer 0: the embedding row, a constant) -> q, k, v
      for (int t : distribute(M_QKV, T_QKV, l)) {
        const MatGeom& m = g.mat[M_QKV];
        const int64_t p0 = s.tasks[t].a[0] * m.Rt, p1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
        if (l > 0) acc(t, B_XRES, 0, H, false, l);
        qkv_writes(t, l, p0, p1, v);
      }
      // attention: one task per (kv head, split) ...
      for (int gh = 0; gh < NKV; ++gh)
        for (int j = 0; j < S; ++j) {
          const int t = task(T_ATTN, l, (gh * S + j) % C);
          s.tasks[t].a[0] = gh;
          s.tasks[t].a[1] = j;
          acc(t, B_QKV, gh * gw, gh * gw + (int64_t)G * hd, false, v);
          if (j == S - 1) acc(t, B_QKV, gh * gw + (int64_t)G * hd, (gh + 1) * gw, false, v);
          acc(t, B_PART, (int64_t)(gh * S + j) * ps, (int64_t)(gh * S + j + 1) * ps, true, v);
        }
      // ... then one LSE merge per query head, queued after every attention
      // task of the layer, spread over the CTAs of its kv head's splits.  It
      // reads the head's acc words of every split and the 4-word vector that
      // holds the head's (m, l) pair.
      for (int gh = 0; gh < NKV; ++gh)
        for (int hh = 0; hh < G; ++hh) {
          const int t = task(T_COMBINE, l, (gh * S + hh * std::max(1, S / G)) % C);
          s.tasks[t].a[0] = gh;
          s.tasks[t].a[1] = hh;
          for (int j = 0; j < S; ++j) {
            const int64_t sb = (int64_t)(gh * S + j) * ps;
            acc(t, B_PART, sb + (int64_t)hh * hd, sb + (int64_t)(hh + 1) * hd, false, v);
            acc(t, B_PART, sb + (int64_t)G * hd + (hh / 2) * 4, sb + (int64_t)G * hd + (hh / 2) * 4 + 4, false, v);
          }
          acc(t, B_O, (int64_t)(gh * G + hh) * hd, (int64_t)(gh * G + hh + 1) * hd, true, v);
        }
      // O projection: x_mid = x_res (layer 0: embedding) + o Wo^T
      for (int t : distribute(M_O, T_OPROJ, l)) {
        const MatGeom& m = g.mat[M_O];
        const int64_t r0 = s.tasks[t].a[0] * m.Rt, r1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
        acc(t, B_O, 0, qd, false, v);
        if (l > 0) acc(t, B_XRES, r0, r1, false, l);
        acc(t, B_XMID, r0, r1, true, v);
      }
      // gate/up + SwiGLU: a = silu(g) * u of rmsnorm(x_mid)
      for (int t : distribute(M_GU, T_GATEUP, l)) {
        const MatGeom& m = g.mat[M_GU];
        const int64_t p0 = s.tasks[t].a[0] * m.Rt, p1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
        acc(t, B_XMID, 0, H, false, v);
        acc(t, B_A, p0 / 2, (p1 + 1) / 2, true, v);
      }
      // down: x_res = x_mid + a Wd^T
      for (int t : distribute(M_DOWN, T_DOWN, l)) {
        const MatGeom& m = g.mat[M_DOWN];
        const int64_t r0 = s.tasks[t].a[0] * m.Rt, r1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
        acc(t, B_A, 0, F, false, v);
        acc(t, B_XMID, r0, r1, false, v);
        acc(t, B_XRES, r0, r1, true, v);
      }
    }

    s.body_len.resize(C);
    for (int q = 0; q < C; ++q) s.body_len[q] = (int)s.queues[q].size();

    // LM head (skipped by prefill).  LM task k also writes the (value,
    // index) of its rows' largest logit to pair k of the argmax buffer.
    const std::vector<int> lm = distribute(M_LM, T_LMHEAD, L - 1);
    s.buffers[B_AMAX] = {(int64_t)lm.size() * 2, BUF_OUTPUT};
    for (size_t k = 0; k < lm.size(); ++k) {
      const int t = lm[k];
      const MatGeom& m = g.mat[M_LM];
      const int64_t r0 = s.tasks[t].a[0] * m.Rt, r1 = std::min<int64_t>(s.tasks[t].a[1] * m.Rt, m.rows);
      s.tasks[t].a[2] = (int64_t)k;
      acc(t, B_XRES, 0, H, false, L);
      acc(t, B_LOGITS, r0, r1, true, 0);
      acc(t, B_AMAX, (int64_t)k * 2, (int64_t)k * 2 + 2, true, 0);
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
  const int64_t T = (int64_t)s.tasks.size(), NQ = (int64_t)s.queues.size(),
                NB = (int64_t)s.buffers.size();
  const int32_t V = s.versions;
  if ((int64_t)s.body_len.size() != NQ) return fail("body_len size differs from queue count");
  if (V < 1 || V > kMaxVersions) return fail(fmt_msg("versions per step %lld outside [1, %lld]", V, kMaxVersions));
  for (int64_t b = 0; b < NB; ++b) {
    const Buffer& B = s.buffers[b];
    if (B.size <= 0 || B.kind < BUF_TAGGED || B.kind > BUF_STATE)
      return fail(fmt_msg("buffer %lld: bad size or kind", b));
  }

  // ---- referential integrity ------------------------------------------
  for (int64_t t = 0; t < T; ++t) {
    const Task& k = s.tasks[t];
    if (k.type < 0 || k.type >= T_NUM_TYPES) return fail(fmt_msg("task %lld: bad type", t));
    if (k.queue < 0 || k.queue >= NQ) return fail(fmt_msg("task %lld: bad queue %lld", t, k.queue));
    bool writes = false;
    for (const Access& a : k.acc) {
      if (a.buffer < 0 || a.buffer >= NB) return fail(fmt_msg("task %lld: bad buffer", t));
      if (a.lo < 0 || a.hi <= a.lo || a.hi > s.buffers[a.buffer].size)
        return fail(fmt_msg("task %lld: access [%lld, %lld) out of its buffer", t, a.lo, a.hi));
      const bool tagged = s.buffers[a.buffer].kind == BUF_TAGGED;
      if (tagged ? (a.version < 1 || a.version > V) : a.version != 0)
        return fail(fmt_msg("task %lld: version %lld invalid for buffer %lld", t, a.version, a.buffer));
      writes |= a.write != 0;
    }
    if (!writes) return fail(fmt_msg("task %lld writes nothing (unreachable work)", t));
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
  for (int64_t t = 0; t < T; ++t)
    if (lane_of[t] == -1) return fail(fmt_msg("task %lld not in its queue", t));
  std::vector<char> in_body(T, 0);
  for (int64_t q = 0; q < NQ; ++q)
    for (int i = 0; i < s.body_len[q]; ++i) in_body[s.queues[q][i]] = 1;

  // ---- versions: one writer per element and version, every version whole --
  // writers[b][v]: write accesses of version v to tagged buffer b, by lo
  struct W { int64_t lo, hi; int32_t task; };
  std::vector<std::vector<std::vector<W>>> writers(NB);
  for (int64_t b = 0; b < NB; ++b)
    if (s.buffers[b].kind == BUF_TAGGED) writers[b].resize(V + 1);
  for (int64_t t = 0; t < T; ++t)
    for (const Access& a : s.tasks[t].acc)
      if (a.write && s.buffers[a.buffer].kind == BUF_TAGGED) {
        if (!in_body[t])
          return fail(fmt_msg("task %lld writes tagged buffer %lld outside the prefill body", t, a.buffer));
        writers[a.buffer][a.version].push_back({a.lo, a.hi, (int32_t)t});
      }
  for (int64_t b = 0; b < NB; ++b) {
    if (s.buffers[b].kind != BUF_TAGGED) continue;
    for (int32_t v = 1; v <= V; ++v) {
      auto& w = writers[b][v];
      std::sort(w.begin(), w.end(), [](const W& x, const W& y) { return x.lo < y.lo; });
      int64_t end = 0;
      for (const W& x : w) {
        if (x.lo < end)
          return fail(fmt_msg("buffer %lld version %lld: element %lld has two writers", b, v, x.lo));
        if (x.lo > end)
          return fail(fmt_msg("buffer %lld version %lld: element %lld is never written", b, v, end));
        end = x.hi;
      }
      if (end < s.buffers[b].size)
        return fail(fmt_msg("buffer %lld version %lld: element %lld is never written", b, v, end));
    }
  }
  // writers of version v overlapping [lo, hi), in element order
  auto overlapping = [&](int32_t b, int32_t v, int64_t lo, int64_t hi, auto&& fn) {
    const auto& w = writers[b][v];
    auto it = std::upper_bound(w.begin(), w.end(), lo, [](int64_t x, const W& y) { return x < y.lo; });
    if (it != w.begin()) --it;
    for (; it != w.end() && it->lo < hi; ++it)
      if (it->hi > lo) fn(*it);
  };

  // ---- acyclicity of queue order + writer -> reader edges ---------------
  std::vector<std::vector<int32_t>> preds(T);   // writers a task waits for
  std::vector<std::vector<int32_t>> succ(T);
  std::vector<int32_t> indeg(T, 0);
  auto edge = [&](int32_t a, int32_t b) {
    succ[a].push_back(b);
    indeg[b]++;
  };
  for (int64_t q = 0; q < NQ; ++q)
    for (size_t i = 1; i < s.queues[q].size(); ++i) edge(s.queues[q][i - 1], s.queues[q][i]);
  for (int64_t t = 0; t < T; ++t) {
    for (const Access& a : s.tasks[t].acc)
      if (!a.write && s.buffers[a.buffer].kind == BUF_TAGGED)
        overlapping(a.buffer, a.version, a.lo, a.hi, [&](const W& w) {
          if (w.task != t) preds[t].push_back(w.task);
        });
    auto& p = preds[t];
    std::sort(p.begin(), p.end());
    p.erase(std::unique(p.begin(), p.end()), p.end());
    for (int32_t w : p) edge(w, (int32_t)t);
  }
  // a task that reads its own write of the version it waits for never starts
  for (int64_t t = 0; t < T; ++t)
    for (const Access& a : s.tasks[t].acc)
      if (!a.write && s.buffers[a.buffer].kind == BUF_TAGGED) {
        bool self = false;
        overlapping(a.buffer, a.version, a.lo, a.hi, [&](const W& w) { self |= w.task == t; });
        if (self) return fail(fmt_msg("task %lld waits for its own write", t));
      }
  std::vector<int32_t> topo;
  topo.reserve(T);
  {
    std::vector<int32_t> deg = indeg;
    for (int64_t t = 0; t < T; ++t)
      if (!deg[t]) topo.push_back((int32_t)t);
    for (size_t i = 0; i < topo.size(); ++i)
      for (int32_t b : succ[topo[i]])
        if (--deg[b] == 0) topo.push_back(b);
    if ((int64_t)topo.size() != T) {
      for (int64_t t = 0; t < T; ++t)
        if (deg[t]) return fail(fmt_msg("dependency cycle through task %lld", t));
    }
  }
  // prefill body: body tasks never wait for skipped work
  for (int64_t t = 0; t < T; ++t)
    if (in_body[t])
      for (int32_t w : preds[t])
        if (!in_body[w]) return fail(fmt_msg("body task %lld waits on skipped task %lld", t, w));

  // ---- deadlock: run the queues to a fixpoint ----------------------------
  {
    std::vector<int32_t> missing(T);
    for (int64_t t = 0; t < T; ++t) missing[t] = (int32_t)preds[t].size();
    std::vector<std::vector<int32_t>> readers(T);
    for (int64_t t = 0; t < T; ++t)
      for (int32_t w : preds[t]) readers[w].push_back((int32_t)t);
    std::vector<size_t> head(NQ, 0);
    bool progress = true;
    while (progress) {
      progress = false;
      for (int64_t q = 0; q < NQ; ++q)
        while (head[q] < s.queues[q].size() && missing[s.queues[q][head[q]]] == 0) {
          for (int32_t r : readers[s.queues[q][head[q]]]) missing[r]--;
          ++head[q];
          progress = true;
        }
    }
    for (int64_t q = 0; q < NQ; ++q)
      if (head[q] < s.queues[q].size())
        return fail(fmt_msg("deadlock: queue %lld stalls at task %lld", q, s.queues[q][head[q]]));
  }

  // ---- happens-before: vector clocks over the queues ---------------------
  const int64_t Wd = NQ;
  std::vector<int32_t> vc((size_t)T * Wd, 0);
  {
    std::vector<int32_t> prev_in_lane(T, -1);
    for (int64_t q = 0; q < NQ; ++q)
      for (size_t i = 1; i < s.queues[q].size(); ++i) prev_in_lane[s.queues[q][i]] = s.queues[q][i - 1];
    for (int32_t t : topo) {
      int32_t* v = &vc[(size_t)t * Wd];
      if (prev_in_lane[t] >= 0) std::memcpy(v, &vc[(size_t)prev_in_lane[t] * Wd], Wd * sizeof(int32_t));
      for (int32_t p : preds[t]) {
        const int32_t* pv = &vc[(size_t)p * Wd];
        for (int64_t i = 0; i < Wd; ++i) v[i] = std::max(v[i], pv[i]);
      }
      v[lane_of[t]] = lane_pos[t];
    }
  }
  auto hb = [&](int32_t a, int32_t b) { return vc[(size_t)b * Wd + lane_of[a]] >= lane_pos[a]; };

  // tagged buffers: writers of consecutive versions ordered (so the whole
  // chain is), and every reader of v finished before the writer of v + 1
  for (int64_t b = 0; b < NB; ++b) {
    if (s.buffers[b].kind != BUF_TAGGED) continue;
    for (int32_t v = 1; v < V; ++v)
      for (const W& w : writers[b][v]) {
        bool ok = true;
        int32_t bad = -1;
        overlapping((int32_t)b, v + 1, w.lo, w.hi, [&](const W& n) {
          if (ok && n.task != w.task && !hb(w.task, n.task)) { ok = false; bad = n.task; }
        });
        if (!ok)
          return fail(fmt_msg("buffer %lld: writer %lld of a version not ordered before writer %lld of the next", b, w.task, bad));
      }
  }
  for (int64_t t = 0; t < T; ++t)
    for (const Access& a : s.tasks[t].acc) {
      if (a.write || s.buffers[a.buffer].kind != BUF_TAGGED || a.version == V) continue;
      bool ok = true;
      int32_t bad = -1;
      overlapping(a.buffer, a.version + 1, a.lo, a.hi, [&](const W& n) {
        if (ok && n.task != t && !hb((int32_t)t, n.task)) { ok = false; bad = n.task; }
      });
      if (!ok)
        return fail(fmt_msg("buffer %lld: reader %lld may find the next version written by %lld", a.buffer, t, bad));
    }
  // tag aliasing: when a reader starts, the words it polls are at most
  // kMaxTagGap versions behind.  A word holds at least the newest version
  // whose writer happened before the reader's queue predecessor finished
  // (writers are chained by version), else the previous step's last one.
  for (int64_t t = 0; t < T; ++t) {
    const int32_t prev = lane_pos[t] > 1 ? s.queues[lane_of[t]][lane_pos[t] - 2] : -1;
    for (const Access& a : s.tasks[t].acc) {
      if (a.write || s.buffers[a.buffer].kind != BUF_TAGGED || a.version <= kMaxTagGap) continue;
      bool ok = false;
      for (int32_t u = a.version - 1; u >= a.version - kMaxTagGap && !ok && prev >= 0; --u) {
        bool all = true;
        overlapping(a.buffer, u, a.lo, a.hi, [&](const W& w) { all = all && hb(w.task, prev); });
        ok = all;
      }
      if (!ok)
        return fail(fmt_msg("buffer %lld: reader %lld may find a version %lld or more behind (tags alias)",
                            a.buffer, t, kTagPeriod));
    }
  }
  // untagged buffers: every write ordered against every overlapping access
  for (int64_t b = 0; b < NB; ++b) {
    if (s.buffers[b].kind == BUF_TAGGED) continue;
    struct Acc { int64_t lo, hi; int32_t task; int32_t write; };
    std::vector<Acc> v;
    for (int64_t t = 0; t < T; ++t)
      for (const Access& a : s.tasks[t].acc)
        if (a.buffer == b) v.push_back({a.lo, a.hi, (int32_t)t, a.write});
    std::sort(v.begin(), v.end(), [](const Acc& x, const Acc& y) { return x.lo < y.lo; });
    for (size_t i = 0; i < v.size(); ++i) {
      for (size_t j = i + 1; j < v.size() && v[j].lo < v[i].hi; ++j) {
        if (!(v[i].write || v[j].write) || v[i].task == v[j].task) continue;
        if (!hb(v[i].task, v[j].task) && !hb(v[j].task, v[i].task))
          return fail(fmt_msg("race on buffer %lld between tasks %lld and %lld", b, v[i].task, v[j].task));
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
  ok.msg = fmt_msg("accepted: %lld tasks, %lld queues, %lld versions", T, NQ, V);
  return ok;
}

// ------------------------------------------------------------ serialisation

std::vector<int64_t> serialize(const Schedule& s) {
  int64_t na = 0, ni = 0;
  for (const Task& t : s.tasks) na += (int64_t)t.acc.size();
  for (const auto& q : s.queues) ni += (int64_t)q.size();
  std::vector<int64_t> o;
  o.reserve(8 + s.buffers.size() * 2 + s.tasks.size() * 9 + na * 5 + s.queues.size() * 3 + ni);
  o.insert(o.end(), {0x414D4B53, 2, (int64_t)s.tasks.size(), (int64_t)s.queues.size(),
                     (int64_t)s.buffers.size(), na, ni, s.versions});
  for (const Buffer& b : s.buffers) o.insert(o.end(), {b.size, b.kind});
  int64_t ab = 0;
  for (const Task& t : s.tasks) {
    o.insert(o.end(), {t.type, t.layer, t.queue, ab, (int64_t)t.acc.size(), t.a[0], t.a[1], t.a[2], t.a[3]});
    ab += (int64_t)t.acc.size();
  }
  for (const Task& t : s.tasks)
    for (const Access& a : t.acc) o.insert(o.end(), {a.buffer, a.lo, a.hi, a.write, a.version});
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
  if (n < 8 || w[0] != 0x414D4B53 || w[1] != 2) return bad("not a serialised schedule");
  const int64_t nt = w[2], nq = w[3], nb = w[4], na = w[5], ni = w[6], nv = w[7];
  const int64_t lim = (int64_t)1 << 31;
  for (int64_t v : {nt, nq, nb, na, ni, nv})
    if (v < 0 || v >= lim) return bad("schedule header sizes out of range");
  const int64_t need = 8 + nb * 2 + nt * 9 + na * 5 + nq * 3 + ni;
  if ((int64_t)n != need) return bad("schedule length does not match its header");
  auto fits32 = [](int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; };
  const int64_t* p = w + 8;
  Schedule s;
  s.versions = (int32_t)nv;
  s.buffers.resize(nb);
  for (auto& b : s.buffers) {
    b.size = p[0];
    if (!fits32(p[1])) return bad("bad buffer kind");
    b.kind = (int32_t)p[1];
    p += 2;
  }
  const int64_t* tasks = p;
  p += nt * 9;
  const int64_t* accs = p;
  p += na * 5;
  s.tasks.resize(nt);
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t* r = tasks + t * 9;
    for (int i = 0; i < 3; ++i)
      if (!fits32(r[i])) return bad("task field out of range");
    Task& k = s.tasks[t];
    k.type = (int32_t)r[0];
    k.layer = (int32_t)r[1];
    k.queue = (int32_t)r[2];
    if (r[3] < 0 || r[4] < 0 || r[3] + r[4] > na) return bad("task access range out of bounds");
    for (int64_t i = 0; i < r[4]; ++i) {
      const int64_t* ar = accs + (r[3] + i) * 5;
      if (!fits32(ar[0]) || !fits32(ar[3]) || !fits32(ar[4])) return bad("bad access");
      k.acc.push_back({(int32_t)ar[0], ar[1], ar[2], (int32_t)ar[3], (int32_t)ar[4]});
    }
    for (int i = 0; i < 4; ++i) k.a[i] = r[5 + i];
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

// ------------------------------------------------------------- requeue

bool requeue(const Schedule& own, const Schedule& given, Schedule* out, std::string* why) {
  auto bad = [&](const std::string& m) {
    *why = m;
    return false;
  };
  if (given.tasks.size() != own.tasks.size())
    return bad(fmt_msg("the schedule has %lld tasks, the model's lowering %lld", (long long)given.tasks.size(),
                       (long long)own.tasks.size()));
  if (given.queues.size() != own.queues.size() || given.body_len.size() != own.queues.size())
    return bad(fmt_msg("the schedule has %lld queues, the launch %lld CTAs", (long long)given.queues.size(),
                       (long long)own.queues.size()));
  // the lowering's task with the same type, layer and parameters
  using Key = std::array<int64_t, 6>;
  auto key = [](const Task& t) { return Key{t.type, t.layer, t.a[0], t.a[1], t.a[2], t.a[3]}; };
  std::map<Key, int32_t> by_key;
  for (size_t i = 0; i < own.tasks.size(); ++i)
    if (!by_key.emplace(key(own.tasks[i]), (int32_t)i).second) return bad("the lowering has duplicate tasks");
  std::vector<int32_t> map_to(given.tasks.size(), -1);
  std::vector<char> used(own.tasks.size(), 0);
  for (size_t i = 0; i < given.tasks.size(); ++i) {
    auto it = by_key.find(key(given.tasks[i]));
    if (it == by_key.end()) return bad(fmt_msg("task %lld is not a task of this model's lowering", (long long)i));
    if (used[it->second]) return bad(fmt_msg("task %lld appears twice", (long long)i));
    used[it->second] = 1;
    map_to[i] = it->second;
  }
  Schedule r;
  r.buffers = own.buffers;
  r.versions = own.versions;
  r.tasks = own.tasks;
  r.queues.assign(given.queues.size(), {});
  r.body_len = given.body_len;
  std::vector<char> queued(own.tasks.size(), 0);
  for (size_t q = 0; q < given.queues.size(); ++q) {
    const auto& items = given.queues[q];
    const int body = given.body_len[q];
    if (body < 0 || body > (int)items.size()) return bad(fmt_msg("queue %lld: bad body length", (long long)q));
    for (size_t i = 0; i < items.size(); ++i) {
      const int32_t gt = items[i];
      if (gt < 0 || gt >= (int32_t)given.tasks.size()) return bad(fmt_msg("queue %lld: bad task id", (long long)q));
      const int32_t t = map_to[gt];
      if (queued[t]) return bad(fmt_msg("queue %lld: a task is queued twice", (long long)q));
      queued[t] = 1;
      const bool lm = r.tasks[t].type == T_LMHEAD;
      if (lm != ((int)i >= body))
        return bad(fmt_msg("queue %lld: LM-head tasks must follow the body, and only they", (long long)q));
      r.tasks[t].queue = (int32_t)q;
      r.queues[q].push_back(t);
    }
  }
  for (size_t t = 0; t < queued.size(); ++t)
    if (!queued[t]) return bad(fmt_msg("task %lld of the lowering is in no queue", (long long)t));
  *out = std::move(r);
  return true;
}

}  // namespace amk
