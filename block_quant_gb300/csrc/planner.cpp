// RaggedShard layout planner and the derived per-shard work tables.
//
// Problem (veScale-FSDP, feynmanwiki walkthrough, paper section 5): the tensors
// of one communication group share a buffer of V equal local shards of size S;
// each tensor is one contiguous interval, intervals never overlap, padding sits
// only between tensors, and a device boundary may fall inside a tensor only at a
// multiple of the tensor's atomic block g from its start.  Minimise S.
//
// Heuristic (bud-325 summary, Key claims / Method; walkthrough, section 5,
// Algorithm 1): default tensor order; a feasibility check per candidate S (the
// pages' DP over "fewest shards holding the first j blocks", monotone in j); S
// restricted to multiples of L = lcm(alpha, g of the tensors assumed to contain a
// whole shard, "Case 3"); those sets taken as prefixes of the tensors sorted by
// size; binary search over the multiples of L.
//
// Feasibility here is earliest-fit: each tensor starts at the smallest admissible
// offset not before the previous tensor's end.  Padding may be inserted anywhere
// between tensors, so an earlier end never hurts the tensors that follow and the
// greedy placement exists iff the DP's final shard count is at most V.
#include <algorithm>
#include <cstring>
#include <numeric>

#include "bq_internal.h"

namespace bq {
namespace {

constexpr int64_t kMaxExtent = int64_t(1) << 61;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// smallest admissible start >= e, or -1 when the tensor cannot end inside V*S
int64_t earliest_start(int64_t e, int64_t n, int64_t g, int64_t S, int64_t V, int64_t align) {
  const int64_t total = V * S;
  int64_t s = round_up(e, align);
  for (;;) {
    if (s + n > total) return -1;
    const int64_t next_boundary = (s / S + 1) * S;
    if (next_boundary >= s + n) return s;  // lies inside one shard
    const int64_t miss = (next_boundary - s) % g;
    if (miss != 0) {  // that boundary would split a block: slide until it does not
      s = round_up(s + miss, align);
      continue;
    }
    if (next_boundary + S < s + n && S % g != 0) {  // two boundaries inside, S not a block multiple
      s = round_up(next_boundary, align);
      continue;
    }
    return s;
  }
}

bool place_all(const std::vector<int64_t>& n, const std::vector<int64_t>& g, const std::vector<int>& ord, int64_t S,
               int64_t V, int64_t align, std::vector<int64_t>* starts) {
  int64_t end = 0;
  for (const int i : ord) {
    const int64_t s = earliest_start(end, n[i], g[i], S, V, align);
    if (s < 0) return false;
    if (starts) (*starts)[i] = s;
    end = s + n[i];
  }
  return true;
}

int64_t tiles_in(const Tensor& t, int64_t len) {
  if (t.one_d()) return ceil_div(len, 128);
  return ceil_div(len / t.cols, 128) * ceil_div(t.cols, 128);
}

int64_t tiles32_in(const Tensor& t, int64_t len) {
  if (t.one_d()) return ceil_div(len, 32);
  return ceil_div(len / t.cols, 32) * ceil_div(t.cols, 32);
}

int64_t adam_blocks_in(const Tensor& t, int64_t len) {
  if (t.adam_kind == BQ_OPT_MUON) return 0;
  if (t.adam_kind == BQ_ADAM_TILE32) return tiles32_in(t, len);
  return t.adam_kind == BQ_ADAM_FLAT256 ? ceil_div(len, 256) : tiles_in(t, len);
}

}  // namespace
}  // namespace bq

using namespace bq;

extern "C" int bq_plan(const bq_tensor_desc* desc, int n, int V, const bq_plan_opts* opts, bq_layout** out) {
  if (!out) return set_error(BQ_EINVAL, "bq_plan: out is NULL");
  *out = nullptr;
  if (!desc || n <= 0 || V < 1) return set_error(BQ_EINVAL, "bq_plan: need n >= 1 descriptors and V >= 1");
  const int64_t alpha = opts ? opts->alpha : 128;
  const int64_t align = opts ? opts->start_align : 16;
  if (alpha < 1 || align < 1) return set_error(BQ_EINVAL, "bq_plan: alpha and start_align must be >= 1");
  const int order_kind = opts ? opts->order : 0;
  if (order_kind < 0 || order_kind > 2) return set_error(BQ_EINVAL, "bq_plan: order must be 0, 1 or 2");

  auto L = new bq_layout();
  L->V = V;
  L->alpha = alpha;
  L->start_align = align;
  std::vector<int64_t> ns(n), gs(n);
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    const bq_tensor_desc& d = desc[i];
    Tensor t{d.rows, d.cols, d.g, 0, d.adam_kind, d.fp8 ? 1 : 0};
    std::string bad;
    if (t.rows < 1 || t.cols < 0 || t.g < 1 || t.cols > kMaxExtent / std::max<int64_t>(t.rows, 1))
      bad = "bad shape or granularity";
    else if (t.adam_kind != BQ_ADAM_FLAT256 && t.adam_kind != BQ_ADAM_TILE128 && t.adam_kind != BQ_OPT_MUON &&
             t.adam_kind != BQ_ADAM_TILE32)
      bad = "unknown adam_kind";
    else if (t.adam_kind == BQ_ADAM_TILE32 && (t.fp8 || t.g % (t.one_d() ? 32 : 32 * t.cols)))
      bad = "32x32 Adam tiles need g to be whole 32-row bands and take no FP8 staging";
    else if (t.adam_kind == BQ_ADAM_TILE32 && !t.one_d() && (t.cols % 8 || t.cols > (int64_t(1) << 23)))
      bad = "2-D tensors with 32x32 Adam tiles need cols % 8 == 0 and cols <= 2^23";
    else if (t.adam_kind == BQ_OPT_MUON && (t.rows < 2 || t.fp8))
      bad = "Muon tensors are 2-D and take no FP8 staging";
    else if (t.adam_kind == BQ_ADAM_FLAT256 && t.g % 256)
      bad = "FLAT256 Adam blocks need g % 256 == 0";
    else if (t.adam_kind == BQ_ADAM_TILE128 && t.g % t.band())
      bad = "128x128 Adam tiles need g to be whole 128-row bands";
    else if (t.fp8 && t.g % t.band())
      bad = "128x128 FP8 tiles need g to be whole 128-row bands";
    else if (!t.one_d() && (t.fp8 || t.adam_kind == BQ_ADAM_TILE128) && t.cols % 8)
      bad = "2-D tensors with FP8 or 128x128 Adam tiles need cols % 8 == 0";
    else if (!t.one_d() && (t.fp8 || t.adam_kind == BQ_ADAM_TILE128) && t.cols > (int64_t(1) << 23))
      bad = "2-D tensors with FP8 or 128x128 Adam tiles need cols <= 2^23";
    if (!bad.empty()) {
      delete L;
      return set_error(BQ_EINVAL, "bq_plan: tensor " + std::to_string(i) + ": " + bad);
    }
    t.numel = t.rows * t.cols;
    ns[i] = t.numel;
    gs[i] = t.g;
    total += t.numel;
    if (total > kMaxExtent) {
      delete L;
      return set_error(BQ_EINVAL, "bq_plan: group too large");
    }
    L->tensors.push_back(t);
  }

  const int64_t base_cap = round_up(total + int64_t(n) * align, alpha);
  if (base_cap > kMaxExtent / V) {
    delete L;
    return set_error(BQ_EINVAL, "bq_plan: V * S would overflow");
  }
  std::vector<int> by_size(n);
  std::iota(by_size.begin(), by_size.end(), 0);
  std::stable_sort(by_size.begin(), by_size.end(), [&](int a, int b) { return ns[a] > ns[b]; });

  // placement order (walkthrough, paper section 5: default, sorted by block size,
  // sorted by shape): 0 = as given; 1 = atomic block size g, largest first;
  // 2 = shape, rows then columns, largest first (equal shapes become neighbours);
  // ties keep the given order
  std::vector<int> ord(n);
  std::iota(ord.begin(), ord.end(), 0);
  if (order_kind == 1)
    std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return gs[a] > gs[b]; });
  else if (order_kind == 2)
    std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) {
      const Tensor &x = L->tensors[a], &y = L->tensors[b];
      return x.rows != y.rows ? x.rows > y.rows : x.cols > y.cols;
    });
  auto feasible = [&](int64_t S) { return place_all(ns, gs, ord, S, V, align, nullptr); };
  int64_t best = -1, best_k = -1;
  int64_t Lk = alpha;
  for (int k = 0; k <= n; ++k) {
    if (k > 0) {
      const int64_t g = gs[by_size[k - 1]];
      const int64_t q = Lk / std::gcd(Lk, g);
      if (q > base_cap / g + 1) break;  // lcm exceeds the cap: no later prefix can win
      Lk = q * g;
    }
    if (Lk > base_cap) break;
    const int64_t lb = std::max(round_up(ceil_div(total, V), Lk), Lk);
    const int64_t cap = round_up(base_cap, Lk);
    int64_t hi = lb;
    while (hi < cap && !feasible(hi)) hi = std::min(hi * 2, cap);
    int64_t lo_j = lb / Lk, hi_j = hi / Lk;
    while (lo_j < hi_j) {
      const int64_t mid = lo_j + (hi_j - lo_j) / 2;
      if (feasible(mid * Lk))
        hi_j = mid;
      else
        lo_j = mid + 1;
    }
    const int64_t Sk = hi_j * Lk;
    if (best < 0 || Sk < best) {
      best = Sk;
      best_k = k;
    }
  }
  L->S = best;
  L->case3 = best_k;
  L->start.assign(n, 0);
  if (best < 0 || !place_all(ns, gs, ord, best, V, align, &L->start)) {
    delete L;
    return set_error(BQ_EINFEASIBLE, "bq_plan: no feasible layout");
  }

  // derived interval and slot tables
  std::vector<int> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return L->start[a] < L->start[b]; });
  int64_t mslot = 0, fslot = 0;
  for (int64_t k = 0; k < V; ++k) {
    L->dev_first.push_back(int64_t(L->intervals.size()));
    L->dev_mslot.push_back(mslot);
    L->dev_fslot.push_back(fslot);
    const int64_t lo_k = k * best, hi_k = lo_k + best;
    for (int i : order) {
      const Tensor& t = L->tensors[i];
      const int64_t lo = std::max(L->start[i], lo_k);
      const int64_t hi = std::min(L->start[i] + t.numel, hi_k);
      if (hi <= lo) continue;
      const int64_t len = hi - lo;
      L->intervals.push_back(Interval{k, i, lo - L->start[i], len, lo - lo_k, mslot, t.fp8 ? fslot : -1});
      mslot += adam_blocks_in(t, len);
      if (t.fp8) fslot += tiles_in(t, len);
    }
  }
  L->dev_first.push_back(int64_t(L->intervals.size()));
  L->dev_mslot.push_back(mslot);
  L->dev_fslot.push_back(fslot);
  L->n_mslots = mslot;
  L->n_fslots = fslot;
  *out = L;
  return BQ_OK;
}

extern "C" void bq_layout_free(bq_layout* layout) { delete layout; }

extern "C" int bq_layout_query(const bq_layout* L, bq_layout_info* info) {
  if (!L || !info) return set_error(BQ_EINVAL, "bq_layout_query: NULL argument");
  int64_t total = 0;
  for (const auto& t : L->tensors) total += t.numel;
  info->V = L->V;
  info->S = L->S;
  info->N = int64_t(L->tensors.size());
  info->n_intervals = int64_t(L->intervals.size());
  info->n_mslots = L->n_mslots;
  info->n_fslots = L->n_fslots;
  info->total_elems = total;
  info->padding_elems = L->V * L->S - total;
  info->export_len = 8 + 7 * info->N + 7 * info->n_intervals + 3 * (L->V + 1);
  info->case3_prefix = L->case3;
  return BQ_OK;
}

// Root of every Muon tensor: longest-processing-time greedy on the nominal
// Newton-Schulz cost 4 m^2 n + 2 m^3 (m, n = smaller, larger dimension) --
// largest first (ties: lower tensor index), each to the least-loaded device
// (ties: lower device index).  A reading of the walkthrough's "load-balanced
// root" (paper section 6.3), which names no rule.
extern "C" int bq_muon_roots(const bq_layout* L, int32_t* roots, size_t n) {
  if (!L || !roots) return set_error(BQ_EINVAL, "bq_muon_roots: NULL argument");
  if (n < L->tensors.size()) return set_error(BQ_ENOSPC, "bq_muon_roots: roots holds fewer than N entries");
  using u128 = unsigned __int128;
  std::vector<std::pair<u128, int>> muon;
  for (size_t i = 0; i < L->tensors.size(); ++i) {
    roots[i] = -1;
    const Tensor& t = L->tensors[i];
    if (t.adam_kind != BQ_OPT_MUON) continue;
    const u128 m = u128(std::min(t.rows, t.cols)), nn = u128(std::max(t.rows, t.cols));
    muon.push_back({4 * m * m * nn + 2 * m * m * m, int(i)});
  }
  std::sort(muon.begin(), muon.end(), [](const std::pair<u128, int>& a, const std::pair<u128, int>& b) {
    return a.first != b.first ? a.first > b.first : a.second < b.second;
  });
  std::vector<u128> load(size_t(L->V), 0);
  for (const auto& c : muon) {
    size_t k = 0;
    for (size_t j = 1; j < load.size(); ++j)
      if (load[j] < load[k]) k = j;
    roots[c.second] = int32_t(k);
    load[k] += c.first;
  }
  return BQ_OK;
}

extern "C" int bq_layout_export(const bq_layout* L, int64_t* buf, size_t n) {
  bq_layout_info info;
  if (int rc = bq_layout_query(L, &info)) return rc;
  if (!buf || n < size_t(info.export_len)) return set_error(BQ_ENOSPC, "bq_layout_export: buffer too small");
  int64_t* p = buf;
  const int64_t hdr[8] = {0x4251, 1, L->V, L->S, info.N, info.n_intervals, L->n_mslots, L->n_fslots};
  for (int64_t x : hdr) *p++ = x;
  for (size_t i = 0; i < L->tensors.size(); ++i) {
    const Tensor& t = L->tensors[i];
    const int64_t row[7] = {L->start[i], t.numel, t.rows, t.cols, t.g, t.adam_kind, t.fp8};
    for (int64_t x : row) *p++ = x;
  }
  for (const Interval& v : L->intervals) {
    const int64_t row[7] = {v.dev, v.tensor, v.t_off, v.len, v.local_off, v.mslot, v.fslot};
    for (int64_t x : row) *p++ = x;
  }
  for (int64_t k = 0; k <= L->V; ++k) {
    *p++ = L->dev_first[k];
    *p++ = L->dev_mslot[k];
    *p++ = L->dev_fslot[k];
  }
  return BQ_OK;
}

// ---------------------------------------------------------------- shard work tables

namespace bq {

void build_shard_tables(const bq_layout& L, int dev_lo, int dev_hi, ShardTables& T) {
  const int64_t S = L.S;
  const int64_t total = int64_t(dev_hi - dev_lo) * S;
  const int64_t mbase = L.dev_mslot[dev_lo], fbase = L.dev_fslot[dev_lo];
  const int64_t first = L.dev_first[dev_lo], last = L.dev_first[dev_hi];

  // ---- pack pieces: intervals and the padding between them, cut at chunk edges
  T.nchunks = ceil_div(total, kPackChunk);
  T.pieces.clear();
  T.chunk_first.assign(size_t(T.nchunks) + 1, 0);
  auto emit = [&](int64_t dst, int64_t len, int32_t tensor, int64_t src) {
    while (len > 0) {
      const int64_t chunk_end = (dst / kPackChunk + 1) * kPackChunk;
      const int64_t n = std::min(len, chunk_end - dst);
      T.pieces.push_back(PackPiece{dst, src, int32_t(n), tensor});
      dst += n;
      src += n;
      len -= n;
    }
  };
  int64_t cursor = 0;
  for (int64_t k = first; k < last; ++k) {
    const Interval& v = L.intervals[k];
    const int64_t pos = (v.dev - dev_lo) * S + v.local_off;
    if (pos > cursor) emit(cursor, pos - cursor, -1, 0);
    emit(pos, v.len, int32_t(v.tensor), v.t_off);
    cursor = pos + v.len;
  }
  if (total > cursor) emit(cursor, total - cursor, -1, 0);
  {
    size_t p = 0;
    for (int64_t c = 0; c < T.nchunks; ++c) {
      while (p < T.pieces.size() && T.pieces[p].dst < c * kPackChunk) ++p;
      T.chunk_first[c] = int32_t(p);
    }
    T.chunk_first[T.nchunks] = int32_t(T.pieces.size());
  }

  // ---- Adam / FP8 groups
  T.flat256.clear();
  T.flat128.clear();
  T.strips.clear();
  T.tiles.clear();
  T.muon.clear();
  T.flat32.clear();
  T.tiles32.clear();
  T.band_tiles.clear();
  T.max_strip_tiles = 0;
  constexpr int64_t kFlatGroupElems = 8192;
  // 1-D tensors (norms, biases: small) go in groups of one block per warp, so
  // their few blocks spread over many CTAs instead of one CTA looping over them
  // (a 1-D Llama-3-70B norm took 13 us as one 8192-element group)
  auto flat_group = [&](const Tensor& t, int64_t block) { return t.one_d() ? 8 * block : kFlatGroupElems; };
  // whole 256-element blocks; 8192 measured 4% faster than 32768 on the GPT-OSS
  // rank-0 slice, where a layer has only a few hundred 32K pieces for 456 CTAs
  constexpr int64_t kBandPiece = 8192;
  for (int64_t k = first; k < last; ++k) {
    const Interval& v = L.intervals[k];
    const Tensor& t = L.tensors[v.tensor];
    const int64_t pos0 = (v.dev - dev_lo) * S + v.local_off;  // local position of element t_off
    const int32_t mslot = int32_t(v.mslot - mbase);
    const int32_t fslot = v.fslot < 0 ? -1 : int32_t(v.fslot - fbase);
    if (t.adam_kind == BQ_OPT_MUON) {
      // Muon: momentum and apply pieces of at most kFlatGroupElems elements
      for (int64_t off = 0; off < v.len; off += kFlatGroupElems)
        T.muon.push_back(PackPiece{pos0 + off, v.t_off + off, int32_t(std::min(kFlatGroupElems, v.len - off)),
                                   int32_t(v.tensor)});
      continue;
    }
    if (t.adam_kind == BQ_ADAM_TILE32) {
      if (t.one_d()) {
        const int64_t gs = flat_group(t, 32);
        for (int64_t off = 0; off < v.len; off += gs)
          T.flat32.push_back(FlatGroup{pos0 + off, int32_t(std::min(gs, v.len - off)), int32_t(mslot + off / 32), -1, 0});
      } else {
        // 32-row bands x 256-column chunks: 8 tiles per group, one warp each
        const int64_t C = t.cols;
        const int64_t r0 = v.t_off / C, r1 = (v.t_off + v.len) / C;
        const int64_t nct = ceil_div(C, 32);
        for (int64_t rb = r0, band = 0; rb < r1; rb += 32, ++band) {
          const int32_t rows = int32_t(std::min<int64_t>(32, r1 - rb));
          const int64_t bpos = pos0 + (rb - r0) * C;
          for (int64_t c0 = 0; c0 < C; c0 += 256)
            T.tiles32.push_back(RegionGroup{bpos + c0, rows, int32_t(C), int32_t(c0),
                                            int32_t(std::min<int64_t>(256, C - c0)),
                                            int32_t(mslot + band * nct + c0 / 32), -1, 0, 0});
        }
      }
      continue;
    }
    if (t.adam_kind == BQ_ADAM_FLAT256 && (t.one_d() || !t.fp8)) {
      const int64_t gs = flat_group(t, 256);
      for (int64_t off = 0; off < v.len; off += gs) {
        const int64_t n = std::min(gs, v.len - off);
        T.flat256.push_back(FlatGroup{pos0 + off, int32_t(n), int32_t(mslot + off / 256),
                                      fslot < 0 ? -1 : int32_t(fslot + off / 128), 0});
      }
    } else if (t.adam_kind == BQ_ADAM_TILE128 && t.one_d()) {
      const int64_t gs = flat_group(t, 128);
      for (int64_t off = 0; off < v.len; off += gs) {
        const int64_t n = std::min(gs, v.len - off);
        T.flat128.push_back(FlatGroup{pos0 + off, int32_t(n), int32_t(mslot + off / 128),
                                      fslot < 0 ? -1 : int32_t(fslot + off / 128), 0});
      }
    } else {
      // 2-D, band-aligned interval: rows [r0, r1) of the tensor
      const int64_t C = t.cols;
      const int64_t r0 = v.t_off / C, r1 = (v.t_off + v.len) / C;
      const int64_t nct = ceil_div(C, 128);
      uint32_t cmul, cshr;
      make_fastdiv(uint32_t(C), &cmul, &cshr);
      for (int64_t rb = r0, band = 0; rb < r1; rb += 128, ++band) {
        const int32_t rows = int32_t(std::min<int64_t>(128, r1 - rb));
        const int64_t bpos = pos0 + (rb - r0) * C;
        const int32_t fband = fslot < 0 ? -1 : int32_t(fslot + band * nct);
        if (t.adam_kind == BQ_ADAM_TILE128) {
          for (int64_t ct = 0; ct < nct; ++ct) {
            const int64_t c0 = ct * 128;
            T.tiles.push_back(RegionGroup{bpos + c0, rows, int32_t(C), int32_t(c0),
                                          int32_t(std::min<int64_t>(128, C - c0)),
                                          int32_t(mslot + band * nct + ct), fband < 0 ? -1 : int32_t(fband + ct),
                                          cmul, cshr});
          }
        } else {
          // FLAT256 Adam + FP8: flat block index of the band start
          const int32_t mband = int32_t(mslot + (rb - r0) * C / 256);
          if (C % 256 == 0) {
            // 256-column strips: every Adam block is one row segment of the strip
            // (C == 256: the strip is its whole band, one flat run; no map needed)
            if (rb == r0 && C > 256) T.maps.push_back(MapInterval{pos0, int32_t(C), int32_t(r1 - r0)});
            for (int64_t c0 = 0; c0 < C; c0 += 256)
              T.strips.push_back(RegionGroup{bpos + c0, rows, int32_t(C), int32_t(c0), 256,
                                             int32_t(mband + c0 / 256), int32_t(fband + c0 / 128), cmul, cshr,
                                             C > 256 ? int32_t(T.maps.size() - 1) : -1, int32_t(rb - r0)});
            T.max_strip_tiles = std::max(T.max_strip_tiles, 2);
          } else {
            // whole 128-row bands (256-element Adam blocks cross rows): Adam over
            // flat pieces of the band (a flat region of one row: rows = 1,
            // width = C = length, no FP8), and one group per FP8 tile for the
            // two-pass quantiser, so a band spreads over many CTAs
            const int64_t nel = int64_t(rows) * C;
            for (int64_t e0 = 0; e0 < nel; e0 += kBandPiece) {
              const int32_t len = int32_t(std::min(kBandPiece, nel - e0));
              T.strips.push_back(RegionGroup{bpos + e0, 1, len, 0, len, int32_t(mband + e0 / 256), -1, 0, 0});
            }
            for (int64_t ct = 0; ct < nct; ++ct) {
              const int64_t c0 = ct * 128;
              T.band_tiles.push_back(RegionGroup{bpos + c0, rows, int32_t(C), int32_t(c0),
                                                 int32_t(std::min<int64_t>(128, C - c0)), 0, int32_t(fband + ct),
                                                 cmul, cshr});
            }
          }
        }
      }
    }
  }
}

// Every element and scale slot a kernel will touch, checked on the host before
// the tables reach the device: returns an empty string when all are in range.
std::string validate_shard_tables(const bq_layout& L, int dev_lo, int dev_hi, const ShardTables& T) {
  const int64_t total = int64_t(dev_hi - dev_lo) * L.S;
  const int64_t nm = L.dev_mslot[dev_hi] - L.dev_mslot[dev_lo];
  const int64_t nf = L.dev_fslot[dev_hi] - L.dev_fslot[dev_lo];
  int64_t cursor = 0;
  for (const PackPiece& p : T.pieces) {
    if (p.dst != cursor || p.len <= 0 || p.dst / kPackChunk != (p.dst + p.len - 1) / kPackChunk)
      return "pack pieces do not tile the shard range";
    if (p.tensor >= int32_t(L.tensors.size()) || p.tensor < -1) return "pack piece tensor out of range";
    if (p.tensor >= 0 && (p.src < 0 || p.src + p.len > L.tensors[p.tensor].numel))
      return "pack piece reads outside its tensor";
    cursor += p.len;
  }
  if (cursor != total) return "pack pieces do not cover the shard range";
  for (int64_t c = 0; c < T.nchunks; ++c)
    if (T.chunk_first[c] > T.chunk_first[c + 1]) return "chunk index not monotone";
  auto flat_ok = [&](const std::vector<FlatGroup>& v, int B) -> bool {
    for (const FlatGroup& g : v) {
      if (g.pos < 0 || g.nelem <= 0 || g.pos + g.nelem > total || g.pos % 8) return false;
      if (g.mslot < 0 || g.mslot + ceil_div(g.nelem, B) > nm) return false;
      if (g.fslot >= 0 && g.fslot + ceil_div(g.nelem, 128) > nf) return false;
    }
    return true;
  };
  if (!flat_ok(T.flat256, 256)) return "flat 256 group out of range";
  if (!flat_ok(T.flat128, 128)) return "flat 128 group out of range";
  if (!flat_ok(T.flat32, 32)) return "flat 32 group out of range";
  for (const RegionGroup& g : T.tiles32) {
    if (g.rows <= 0 || g.rows > 32 || g.width <= 0 || g.width > 256 || g.width % 8 || g.C % 8 || g.pos % 8 ||
        g.pos < 0 || g.c0 % 32 || g.c0 + g.width > g.C)
      return "32x32 tile group shape";
    if (g.pos + int64_t(g.rows - 1) * g.C + g.width > total) return "32x32 tile group reads outside the shard range";
    if (g.mslot < 0 || g.mslot + ceil_div(g.width, 32) > nm) return "32x32 tile slots out of range";
  }
  for (const RegionGroup& g : T.strips) {
    const bool flat = g.width == g.C;
    if (g.rows <= 0 || g.rows > 128 || g.C % 8 || g.width % 8 || g.pos % 8 || g.pos < 0) return "strip shape";
    const int64_t last = flat ? g.pos + int64_t(g.rows) * g.C : g.pos + int64_t(g.rows - 1) * g.C + g.width;
    if (last > total) return "strip reads outside the shard range";
    if (!flat && (g.C % 256 || g.c0 % 256 || g.width != 256 || g.c0 + g.width > g.C)) return "strip columns";
    if (int64_t(g.rows) * g.C >= (int64_t(1) << 31)) return "strip band too large for 32-bit offsets";
    const int64_t mend = flat ? g.mslot + ceil_div(int64_t(g.rows) * g.C, 256)
                              : g.mslot + int64_t(g.rows - 1) * (g.C / 256) + g.width / 256;
    if (g.mslot < 0 || mend > nm) return "strip Adam slots out of range";
    if (g.fslot < 0 && !flat) return "2-D strip without FP8 slots";
    // FP8 regions are 256-column strips (a 256-column tensor's strip is also its
    // whole band, where both readings of the geometry agree)
    if (g.fslot >= 0 && g.width != 256) return "FP8 region that is not a 256-column strip";
    if (g.fslot >= 0 && g.fslot + ceil_div(g.width, 128) > nf) return "strip FP8 slots out of range";
    if (g.fslot >= 0 && ceil_div(g.width, 128) > T.max_strip_tiles) return "strip tile count above the shared-memory bound";
    if (g.tm >= 0) {  // read through its interval's tensor maps: the box origin must be this strip
      if (flat || g.tm >= int32_t(T.maps.size())) return "strip map index";
      const MapInterval& m = T.maps[size_t(g.tm)];
      if (m.C != g.C || g.trow < 0 || g.trow + g.rows > m.rows || m.pos + int64_t(g.trow) * g.C + g.c0 != g.pos)
        return "strip outside its map interval";
    }
  }
  for (const MapInterval& m : T.maps)
    if (m.pos < 0 || m.C <= 0 || m.C % 256 || m.rows <= 0 || m.pos + int64_t(m.rows) * m.C > total)
      return "map interval outside the shard range";
  for (const RegionGroup& g : T.band_tiles) {
    if (g.rows <= 0 || g.rows > 128 || g.width <= 0 || g.width > 128 || g.width % 8 || g.C % 8 || g.pos % 8 ||
        g.pos < 0 || g.c0 + g.width > g.C || (g.width == g.C && g.c0 != 0))
      return "band FP8 tile shape";
    if (g.pos + int64_t(g.rows - 1) * g.C + g.width > total) return "band FP8 tile outside the shard range";
    if (g.fslot < 0 || g.fslot >= nf) return "band FP8 tile slot out of range";
  }
  for (const PackPiece& p : T.muon) {
    if (p.len <= 0 || p.dst < 0 || p.dst + p.len > total) return "Muon piece outside the shard range";
    if (p.tensor < 0 || p.tensor >= int32_t(L.tensors.size()) || L.tensors[p.tensor].adam_kind != BQ_OPT_MUON)
      return "Muon piece of a non-Muon tensor";
    if (p.src < 0 || p.src + p.len > L.tensors[p.tensor].numel) return "Muon piece reads outside its tensor";
  }
  for (const RegionGroup& g : T.tiles) {
    if (g.rows <= 0 || g.rows > 128 || g.width <= 0 || g.width > 128 || g.width % 8 || g.C % 8 || g.pos % 8 ||
        g.pos < 0 || g.c0 + g.width > g.C)
      return "tile shape";
    if (g.pos + int64_t(g.rows - 1) * g.C + g.width > total) return "tile reads outside the shard range";
    if (g.mslot < 0 || g.mslot >= nm || g.fslot >= nf) return "tile slots out of range";
  }
  return std::string();
}

// ---------------------------------------------------------------- groups of shard ranges
// A group is several (layout, [dev_lo, dev_hi)) members stepped by one launch
// per kernel family: every member's tables are built and checked alone, then
// appended with its element, slot and tensor bases added.  Pack pieces are cut
// again at the group's chunk edges, and the alignment gaps between members
// become padding pieces (zeroed by the pack like any padding).

void append_member_tables(const ShardTables& M, const GroupPlace& at, ShardTables& G) {
  auto emit = [&](int64_t dst, int64_t len, int32_t tensor, int64_t src) {
    while (len > 0) {
      const int64_t chunk_end = (dst / kPackChunk + 1) * kPackChunk;
      const int64_t n = std::min(len, chunk_end - dst);
      G.pieces.push_back(PackPiece{dst, src, int32_t(n), tensor});
      dst += n;
      src += n;
      len -= n;
    }
  };
  const int64_t cursor = G.pieces.empty() ? 0 : G.pieces.back().dst + G.pieces.back().len;
  if (at.elem > cursor) emit(cursor, at.elem - cursor, -1, 0);  // gap before the member
  for (const PackPiece& q : M.pieces)
    emit(at.elem + q.dst, q.len, q.tensor < 0 ? -1 : int32_t(q.tensor + at.tensor), q.src);
  auto flat = [&](const std::vector<FlatGroup>& src, std::vector<FlatGroup>& dst) {
    for (FlatGroup g : src) {
      g.pos += at.elem;
      g.mslot += int32_t(at.mslot);
      if (g.fslot >= 0) g.fslot += int32_t(at.fslot);
      dst.push_back(g);
    }
  };
  const int32_t tm0 = int32_t(G.maps.size());  // the member's map intervals start here
  for (MapInterval m : M.maps) {
    m.pos += at.elem;
    G.maps.push_back(m);
  }
  auto region = [&](const std::vector<RegionGroup>& src, std::vector<RegionGroup>& dst, bool mslots) {
    for (RegionGroup g : src) {
      g.pos += at.elem;
      if (mslots) g.mslot += int32_t(at.mslot);
      if (g.fslot >= 0) g.fslot += int32_t(at.fslot);
      if (g.tm >= 0) g.tm += tm0;
      dst.push_back(g);
    }
  };
  flat(M.flat256, G.flat256);
  flat(M.flat128, G.flat128);
  flat(M.flat32, G.flat32);
  region(M.strips, G.strips, true);
  region(M.tiles, G.tiles, true);
  region(M.tiles32, G.tiles32, true);
  region(M.band_tiles, G.band_tiles, false);  // band FP8 tiles carry no Adam slot
  for (PackPiece q : M.muon) {
    q.dst += at.elem;
    q.tensor += int32_t(at.tensor);
    G.muon.push_back(q);
  }
  G.max_strip_tiles = std::max(G.max_strip_tiles, M.max_strip_tiles);
}

void finish_group_tables(int64_t group_total, ShardTables& G) {
  const int64_t cursor = G.pieces.empty() ? 0 : G.pieces.back().dst + G.pieces.back().len;
  for (int64_t dst = cursor; dst < group_total;) {  // trailing gap: padding
    const int64_t n = std::min(group_total - dst, (dst / kPackChunk + 1) * kPackChunk - dst);
    G.pieces.push_back(PackPiece{dst, 0, int32_t(n), -1});
    dst += n;
  }
  G.nchunks = ceil_div(group_total, kPackChunk);
  G.chunk_first.assign(size_t(G.nchunks) + 1, 0);
  size_t p = 0;
  for (int64_t c = 0; c < G.nchunks; ++c) {
    while (p < G.pieces.size() && G.pieces[p].dst < c * kPackChunk) ++p;
    G.chunk_first[c] = int32_t(p);
  }
  G.chunk_first[G.nchunks] = int32_t(G.pieces.size());
}

}  // namespace bq
