// C ABI of libbq: errors, device-table upload, argument validation and dispatch
// to the step kernels.  All compute runs in the CUDA kernels; this file only
// checks arguments, builds integer work tables and launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "bq_internal.h"

namespace bq {

static thread_local std::string g_last_error;

int set_error(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

// true the first time (device, key) is seen in this process: one-time per-device
// set-up such as kernel attributes, which belong to the device they were set on
bool once_per_device(int key) {
  static std::mutex mu;
  static bool done[64][8] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || key < 0 || key >= 8) return true;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev][key]) return false;
  done[dev][key] = true;
  return true;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

}  // namespace bq

using namespace bq;

struct bq_shard {
  const bq_layout* layout;
  int dev_lo, dev_hi;
  int64_t total;           // elements of the shard range
  int64_t nm, nf;          // Adam / FP8 scale slots of the range
  DevTables dev;
  // the strips' tensor maps in the workspace hold the buffers of the last step
  // that wrote them (key); they are rebuilt when the buffers change
  std::vector<MapInterval> maps;
  mutable std::mutex map_mu;
  mutable const void* map_key[4] = {nullptr, nullptr, nullptr, nullptr};
  mutable bool map_ok = false;
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsPlan {
  size_t off_pieces, off_chunks, off_f256, off_f128, off_strips, off_tiles, off_muon, off_f32, off_t32, off_bt,
      off_status, off_maps, bytes;
};

WsPlan ws_plan(const ShardTables& T) {
  WsPlan p;
  size_t o = 0;
  p.off_pieces = o;
  o = align_up(o + T.pieces.size() * sizeof(PackPiece), 256);
  p.off_chunks = o;
  o = align_up(o + T.chunk_first.size() * sizeof(int32_t), 256);
  p.off_f256 = o;
  o = align_up(o + T.flat256.size() * sizeof(FlatGroup), 256);
  p.off_f128 = o;
  o = align_up(o + T.flat128.size() * sizeof(FlatGroup), 256);
  p.off_strips = o;
  o = align_up(o + T.strips.size() * sizeof(RegionGroup), 256);
  p.off_tiles = o;
  o = align_up(o + T.tiles.size() * sizeof(RegionGroup), 256);
  p.off_muon = o;
  o = align_up(o + T.muon.size() * sizeof(PackPiece), 256);
  p.off_f32 = o;
  o = align_up(o + T.flat32.size() * sizeof(FlatGroup), 256);
  p.off_t32 = o;
  o = align_up(o + T.tiles32.size() * sizeof(RegionGroup), 256);
  p.off_bt = o;
  o = align_up(o + T.band_tiles.size() * sizeof(RegionGroup), 256);
  p.off_status = o;  // device error word, zeroed by the upload
  o += 256;
  p.off_maps = o;  // 4 tensor maps per map interval, written by the first step on a set of buffers
  o = align_up(o + T.maps.size() * 4 * kMapBytes, 256);
  p.bytes = o;
  return p;
}

int check_range(const bq_layout* L, int dev_lo, int dev_hi) {
  if (!L) return set_error(BQ_EINVAL, "layout is NULL");
  if (dev_lo < 0 || dev_hi > L->V || dev_lo >= dev_hi)
    return set_error(BQ_EINVAL, "need 0 <= dev_lo < dev_hi <= V");
  for (int64_t k = L->dev_first[dev_lo]; k < L->dev_first[dev_hi]; ++k)
    if (L->intervals[k].local_off % 8)
      return set_error(BQ_EALIGN, "interval local offsets must be multiples of 8 elements (plan with start_align % 8 == 0)");
  if (int64_t(dev_hi - dev_lo) * L->S > (int64_t(1) << 40))
    return set_error(BQ_EINVAL, "shard range too large");
  return BQ_OK;
}

// Stage every table in one host image, copy it with one synchronised copy (the
// image may be freed on return) and make the host shard object pointing at it.
int upload_tables(const ShardTables& T, void* dev_ws, size_t ws_bytes, bq_stream_t stream, const char* who,
                  bq_shard** out) {
  const WsPlan p = ws_plan(T);
  if (ws_bytes < p.bytes) return set_error(BQ_ENOSPC, std::string(who) + ": workspace too small");
  std::vector<unsigned char> img(p.bytes, 0);
  auto put = [&](size_t off, const void* src, size_t n) {
    if (n) std::memcpy(img.data() + off, src, n);
  };
  put(p.off_pieces, T.pieces.data(), T.pieces.size() * sizeof(PackPiece));
  put(p.off_chunks, T.chunk_first.data(), T.chunk_first.size() * sizeof(int32_t));
  put(p.off_f256, T.flat256.data(), T.flat256.size() * sizeof(FlatGroup));
  put(p.off_f128, T.flat128.data(), T.flat128.size() * sizeof(FlatGroup));
  put(p.off_strips, T.strips.data(), T.strips.size() * sizeof(RegionGroup));
  put(p.off_tiles, T.tiles.data(), T.tiles.size() * sizeof(RegionGroup));
  put(p.off_muon, T.muon.data(), T.muon.size() * sizeof(PackPiece));
  put(p.off_f32, T.flat32.data(), T.flat32.size() * sizeof(FlatGroup));
  put(p.off_t32, T.tiles32.data(), T.tiles32.size() * sizeof(RegionGroup));
  put(p.off_bt, T.band_tiles.data(), T.band_tiles.size() * sizeof(RegionGroup));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(dev_ws, img.data(), p.bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(BQ_ECUDA, std::string(who) + ": " + cudaGetErrorString(e));

  auto* sh = new bq_shard();
  auto* base = static_cast<unsigned char*>(dev_ws);
  sh->dev.pieces = reinterpret_cast<const PackPiece*>(base + p.off_pieces);
  sh->dev.chunk_first = reinterpret_cast<const int32_t*>(base + p.off_chunks);
  sh->dev.flat256 = reinterpret_cast<const FlatGroup*>(base + p.off_f256);
  sh->dev.flat128 = reinterpret_cast<const FlatGroup*>(base + p.off_f128);
  sh->dev.strips = reinterpret_cast<const RegionGroup*>(base + p.off_strips);
  sh->dev.tiles = reinterpret_cast<const RegionGroup*>(base + p.off_tiles);
  sh->dev.muon = reinterpret_cast<const PackPiece*>(base + p.off_muon);
  sh->dev.flat32 = reinterpret_cast<const FlatGroup*>(base + p.off_f32);
  sh->dev.tiles32 = reinterpret_cast<const RegionGroup*>(base + p.off_t32);
  sh->dev.band_tiles = reinterpret_cast<const RegionGroup*>(base + p.off_bt);
  sh->dev.nchunks = T.nchunks;
  sh->dev.n_flat256 = int32_t(T.flat256.size());
  sh->dev.n_flat128 = int32_t(T.flat128.size());
  sh->dev.n_strips = int32_t(T.strips.size());
  sh->dev.n_tiles = int32_t(T.tiles.size());
  sh->dev.n_muon = int32_t(T.muon.size());
  sh->dev.n_flat32 = int32_t(T.flat32.size());
  sh->dev.n_tiles32 = int32_t(T.tiles32.size());
  sh->dev.n_band_tiles = int32_t(T.band_tiles.size());
  sh->dev.max_strip_tiles = T.max_strip_tiles;
  sh->dev.status = reinterpret_cast<int*>(base + p.off_status);
  sh->dev.tmaps = base + p.off_maps;
  sh->dev.n_maps = int32_t(T.maps.size());
  sh->maps = T.maps;
  *out = sh;
  return BQ_OK;
}

// Members' element ranges start at multiples of kGroupAlign elements (16-byte
// aligned in every buffer, whole 256-element Adam blocks apart); slots and
// tensors follow one another without gaps.
constexpr int64_t kGroupAlign = 256;

int group_place(const bq_member* members, int n, std::vector<bq_member_place>& pl, bq_group_info& gi) {
  if (!members || n < 1) return set_error(BQ_EINVAL, "bq_group: need at least one member");
  pl.assign(size_t(n), bq_member_place{0, 0, 0, 0});
  int64_t elem = 0, ms = 0, fs = 0, nt = 0, end = 0;
  for (int u = 0; u < n; ++u) {
    const bq_layout* L = members[u].layout;
    const int lo = members[u].dev_lo, hi = members[u].dev_hi;
    if (int rc = check_range(L, lo, hi)) return rc;
    elem = align_up(size_t(end), size_t(kGroupAlign));
    pl[u] = bq_member_place{elem, ms, fs, nt};
    end = elem + int64_t(hi - lo) * L->S;
    ms += L->dev_mslot[hi] - L->dev_mslot[lo];
    fs += L->dev_fslot[hi] - L->dev_fslot[lo];
    nt += int64_t(L->tensors.size());
  }
  if (end > (int64_t(1) << 40) || ms >= (int64_t(1) << 31) || fs >= (int64_t(1) << 31) || nt >= (int64_t(1) << 31))
    return set_error(BQ_EINVAL, "bq_group: group too large (2^40 elements, 2^31 slots or tensors)");
  gi = bq_group_info{end, ms, fs, nt};
  return BQ_OK;
}

int build_group(const bq_member* members, int n, ShardTables& G, bq_group_info& gi) {
  std::vector<bq_member_place> pl;
  if (int rc = group_place(members, n, pl, gi)) return rc;
  for (int u = 0; u < n; ++u) {
    const bq_layout& L = *members[u].layout;
    ShardTables M;
    build_shard_tables(L, members[u].dev_lo, members[u].dev_hi, M);
    const std::string bad = validate_shard_tables(L, members[u].dev_lo, members[u].dev_hi, M);
    if (!bad.empty())
      return set_error(BQ_EINVAL, "bq_group: internal table check of member " + std::to_string(u) + " failed: " + bad);
    append_member_tables(M, GroupPlace{pl[u].elem_base, pl[u].mslot_base, pl[u].fslot_base, pl[u].tensor_base}, G);
  }
  finish_group_tables(gi.elems, G);
  // the concatenation itself: pieces tile [0, elems) inside their chunks
  int64_t cursor = 0;
  for (const PackPiece& q : G.pieces) {
    if (q.dst != cursor || q.len <= 0 || q.dst / kPackChunk != (q.dst + q.len - 1) / kPackChunk)
      return set_error(BQ_EINVAL, "bq_group: internal check failed: pack pieces do not tile the group");
    cursor += q.len;
  }
  if (cursor != gi.elems) return set_error(BQ_EINVAL, "bq_group: internal check failed: pack pieces do not cover the group");
  return BQ_OK;
}

}  // namespace

extern "C" {

const char* bq_strerror(int code) {
  switch (code) {
    case BQ_OK: return "ok";
    case BQ_EINVAL: return "invalid argument";
    case BQ_EINFEASIBLE: return "no feasible layout";
    case BQ_EALIGN: return "misaligned pointer or offset";
    case BQ_ECUDA: return "CUDA error";
    case BQ_ENOSPC: return "buffer or workspace too small";
    case BQ_EDEVICE: return "no usable device";
    default: return "unknown error";
  }
}

const char* bq_last_error(void) { return g_last_error.c_str(); }

int bq_version(void) { return 1; }

int bq_layout_upload_bytes(const bq_layout* L, int dev_lo, int dev_hi, size_t* bytes) {
  if (!bytes) return set_error(BQ_EINVAL, "bq_layout_upload_bytes: bytes is NULL");
  if (int rc = check_range(L, dev_lo, dev_hi)) return rc;
  ShardTables T;
  build_shard_tables(*L, dev_lo, dev_hi, T);
  const std::string bad = validate_shard_tables(*L, dev_lo, dev_hi, T);
  if (!bad.empty()) return set_error(BQ_EINVAL, "bq_layout_upload_bytes: internal table check failed: " + bad);
  *bytes = ws_plan(T).bytes;
  return BQ_OK;
}

int bq_layout_upload(const bq_layout* L, int dev_lo, int dev_hi, void* dev_ws, size_t ws_bytes, bq_stream_t stream,
                     bq_shard** out) {
  if (!out) return set_error(BQ_EINVAL, "bq_layout_upload: out is NULL");
  *out = nullptr;
  if (int rc = check_range(L, dev_lo, dev_hi)) return rc;
  if (!dev_ws || !aligned16(dev_ws)) return set_error(BQ_EALIGN, "bq_layout_upload: workspace NULL or misaligned");
  ShardTables T;
  build_shard_tables(*L, dev_lo, dev_hi, T);
  const std::string bad = validate_shard_tables(*L, dev_lo, dev_hi, T);
  if (!bad.empty()) return set_error(BQ_EINVAL, "bq_layout_upload: internal table check failed: " + bad);
  const int64_t total = int64_t(dev_hi - dev_lo) * L->S;
  const int64_t nm = L->dev_mslot[dev_hi] - L->dev_mslot[dev_lo];
  const int64_t nf = L->dev_fslot[dev_hi] - L->dev_fslot[dev_lo];
  if (int rc = upload_tables(T, dev_ws, ws_bytes, stream, "bq_layout_upload", out)) return rc;
  (*out)->layout = L;
  (*out)->dev_lo = dev_lo;
  (*out)->dev_hi = dev_hi;
  (*out)->total = total;
  (*out)->nm = nm;
  (*out)->nf = nf;
  return BQ_OK;
}

int bq_group_place(const bq_member* members, int n, bq_member_place* place, bq_group_info* info) {
  std::vector<bq_member_place> pl;
  bq_group_info gi;
  if (int rc = group_place(members, n, pl, gi)) return rc;
  if (place)
    for (int u = 0; u < n; ++u) place[u] = pl[u];
  if (info) *info = gi;
  return BQ_OK;
}

int bq_group_upload_bytes(const bq_member* members, int n, size_t* bytes) {
  if (!bytes) return set_error(BQ_EINVAL, "bq_group_upload_bytes: bytes is NULL");
  ShardTables G;
  bq_group_info gi;
  if (int rc = build_group(members, n, G, gi)) return rc;
  *bytes = ws_plan(G).bytes;
  return BQ_OK;
}

int bq_group_upload(const bq_member* members, int n, void* dev_ws, size_t ws_bytes, bq_stream_t stream,
                    bq_shard** out) {
  if (!out) return set_error(BQ_EINVAL, "bq_group_upload: out is NULL");
  *out = nullptr;
  if (!dev_ws || !aligned16(dev_ws)) return set_error(BQ_EALIGN, "bq_group_upload: workspace NULL or misaligned");
  ShardTables G;
  bq_group_info gi;
  if (int rc = build_group(members, n, G, gi)) return rc;
  if (int rc = upload_tables(G, dev_ws, ws_bytes, stream, "bq_group_upload", out)) return rc;
  (*out)->layout = nullptr;
  (*out)->total = gi.elems;
  (*out)->nm = gi.mslots;
  (*out)->nf = gi.fslots;
  return BQ_OK;
}

void bq_shard_free(bq_shard* shard) { delete shard; }

int bq_pack(const bq_shard* sh, const void* const* grad_ptrs, void* dbuf_grad, float scale, int accumulate,
            bq_stream_t stream) {
  if (!sh || !grad_ptrs || !dbuf_grad) return set_error(BQ_EINVAL, "bq_pack: NULL argument");
  if (!aligned16(grad_ptrs) && (reinterpret_cast<uintptr_t>(grad_ptrs) & 7))
    return set_error(BQ_EALIGN, "bq_pack: grad_ptrs must be 8-byte aligned");
  if (!aligned16(dbuf_grad)) return set_error(BQ_EALIGN, "bq_pack: dbuf_grad must be 16-byte aligned");
  return launch_pack(sh->dev, reinterpret_cast<const uint16_t* const*>(grad_ptrs),
                     static_cast<uint16_t*>(dbuf_grad), sh->total, scale, accumulate ? 1 : 0, stream);
}

// The strips' tensor maps for these buffers (grad bf16, master fp32, m, v bytes:
// 8-row x 256-column boxes of each map interval), or NULL, in which case the
// strip kernel copies block by block (the same data).  Built and copied into the
// workspace, on `stream`, when the buffers differ from the last step's.  A step
// being captured into a graph never uses them: a replay must not depend on which
// buffers a later call wrote maps for.
static const void* strip_maps(const bq_shard* sh, const void* grad, const void* master, const void* m,
                              const void* v, bq_stream_t stream) {
  if (sh->dev.n_maps == 0) return nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(sh->map_mu);
  const void* key[4] = {grad, master, m, v};
  if (std::equal(key, key + 4, sh->map_key)) return sh->map_ok ? sh->dev.tmaps : nullptr;
  constexpr int kElem[4] = {2, 4, 1, 1};
  std::vector<unsigned char> img(sh->maps.size() * 4 * kMapBytes);
  bool ok = true;
  for (size_t i = 0; ok && i < sh->maps.size(); ++i)
    for (int k = 0; ok && k < 4; ++k) {
      const MapInterval& mi = sh->maps[i];
      const auto* base = static_cast<const unsigned char*>(key[k]) + mi.pos * kElem[k];
      ok = (reinterpret_cast<uintptr_t>(base) & 15) == 0 &&  // tensor map bases are 16-byte aligned
           encode_map_2d(img.data() + (i * 4 + size_t(k)) * kMapBytes, base, kElem[k], mi.C, mi.rows, 256, 8) == BQ_OK;
    }
  if (ok) ok = cudaMemcpyAsync(sh->dev.tmaps, img.data(), img.size(), cudaMemcpyHostToDevice, s) == cudaSuccess;
  if (!ok) cudaGetLastError();
  std::copy(key, key + 4, sh->map_key);
  sh->map_ok = ok;
  return ok ? sh->dev.tmaps : nullptr;
}

int bq_step_adam8(const bq_shard* sh, const void* grad, float* master, int8_t* m, uint8_t* v, float* m_scale,
                  float* v_scale, const bq_adam_hp* hp, uint8_t* fp8_out, float* fp8_scale, bq_stream_t stream) {
  if (!sh || !grad || !master || !m || !v || !hp) return set_error(BQ_EINVAL, "bq_step_adam8: NULL argument");
  // scale buffers may be NULL only when the range has no slots of that kind
  if (sh->nm > 0 && (!m_scale || !v_scale)) return set_error(BQ_EINVAL, "bq_step_adam8: NULL scale buffer");
  if (fp8_out && !fp8_scale && sh->nf > 0)
    return set_error(BQ_EINVAL, "bq_step_adam8: fp8_out needs fp8_scale");
  if (!fp8_out && fp8_scale) return set_error(BQ_EINVAL, "bq_step_adam8: fp8_scale without fp8_out");
  const void* ptrs[] = {grad, master, m, v, fp8_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return set_error(BQ_EALIGN, "bq_step_adam8: buffers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(m_scale) | reinterpret_cast<uintptr_t>(v_scale) |
       reinterpret_cast<uintptr_t>(fp8_scale)) & 3)
    return set_error(BQ_EALIGN, "bq_step_adam8: scale buffers must be 4-byte aligned");
  AdamArgs a{static_cast<const uint16_t*>(grad), master, m, v, m_scale, v_scale, fp8_out, fp8_scale, *hp,
             sh->dev.status, strip_maps(sh, grad, master, m, v, stream)};
  return launch_adam8(sh->dev, a, stream);
}

int bq_adam_hparams(double lr, double b1, double b2, double eps, int64_t t, bq_adam_hp* out) {
  if (!out) return set_error(BQ_EINVAL, "bq_adam_hparams: out is NULL");
  if (t < 1) return set_error(BQ_EINVAL, "bq_adam_hparams: the step count t starts at 1");
  if (!(b1 >= 0.0 && b1 < 1.0) || !(b2 >= 0.0 && b2 < 1.0))
    return set_error(BQ_EINVAL, "bq_adam_hparams: b1 and b2 must lie in [0, 1)");
  if (!(lr >= 0.0) || !std::isfinite(lr) || !(eps >= 0.0) || !std::isfinite(eps))
    return set_error(BQ_EINVAL, "bq_adam_hparams: lr and eps must be finite and non-negative");
  // fp64 throughout, one rounding to fp32 at the end
  const double bc1 = 1.0 - std::pow(b1, double(t)), bc2 = 1.0 - std::pow(b2, double(t));
  *out = bq_adam_hp{float(lr), float(b1), float(b2), float(eps), float(1.0 - b1), float(1.0 - b2),
                    float(1.0 / bc1), float(1.0 / bc2)};
  return BQ_OK;
}

int bq_quant_fp8(const bq_shard* sh, const float* master, uint8_t* fp8_out, float* fp8_scale, bq_stream_t stream) {
  if (!sh || !master || !fp8_out) return set_error(BQ_EINVAL, "bq_quant_fp8: NULL argument");
  if (!fp8_scale && sh->nf > 0) return set_error(BQ_EINVAL, "bq_quant_fp8: NULL fp8_scale");
  if (!aligned16(master) || !aligned16(fp8_out) || (reinterpret_cast<uintptr_t>(fp8_scale) & 3))
    return set_error(BQ_EALIGN, "bq_quant_fp8: misaligned buffer");
  return launch_quant_fp8(sh->dev, master, fp8_out, fp8_scale, stream);
}

int bq_dequant_fp8(const bq_shard* sh, const uint8_t* fp8, const float* fp8_scale, void* out_bf16, bq_stream_t stream) {
  if (!sh || !fp8 || !out_bf16) return set_error(BQ_EINVAL, "bq_dequant_fp8: NULL argument");
  if (!fp8_scale && sh->nf > 0) return set_error(BQ_EINVAL, "bq_dequant_fp8: NULL fp8_scale");
  if (!aligned16(fp8) || !aligned16(out_bf16) || (reinterpret_cast<uintptr_t>(fp8_scale) & 3))
    return set_error(BQ_EALIGN, "bq_dequant_fp8: misaligned buffer");
  return launch_dequant_fp8(sh->dev, fp8, fp8_scale, static_cast<uint16_t*>(out_bf16), stream);
}

int bq_muon_momentum(const bq_shard* sh, const void* grad, float* mom, float mu, void* const* gather_ptrs,
                     bq_stream_t stream) {
  if (!sh || !grad || !mom || !gather_ptrs) return set_error(BQ_EINVAL, "bq_muon_momentum: NULL argument");
  if (!aligned16(grad) || !aligned16(mom) || (reinterpret_cast<uintptr_t>(gather_ptrs) & 7))
    return set_error(BQ_EALIGN, "bq_muon_momentum: grad and mom 16-byte, gather_ptrs 8-byte aligned");
  return launch_muon_momentum(sh->dev, static_cast<const uint16_t*>(grad), mom, mu,
                              reinterpret_cast<uint16_t* const*>(gather_ptrs), stream);
}

int bq_muon_apply(const bq_shard* sh, float* master, const void* const* update_ptrs, const float* lr,
                  bq_stream_t stream) {
  if (!sh || !master || !update_ptrs || !lr) return set_error(BQ_EINVAL, "bq_muon_apply: NULL argument");
  if (!aligned16(master) || (reinterpret_cast<uintptr_t>(update_ptrs) & 7) || (reinterpret_cast<uintptr_t>(lr) & 3))
    return set_error(BQ_EALIGN, "bq_muon_apply: master 16-byte, update_ptrs 8-byte, lr 4-byte aligned");
  return launch_muon_apply(sh->dev, master, reinterpret_cast<const uint16_t* const*>(update_ptrs), lr, stream);
}

int bq_wait_selftest(int* dev_status, bq_stream_t stream) {
  if (!dev_status || (reinterpret_cast<uintptr_t>(dev_status) & 3))
    return set_error(BQ_EINVAL, "bq_wait_selftest: dev_status NULL or misaligned");
  return launch_wait_selftest(dev_status, stream);
}

int bq_shard_check(const bq_shard* sh, bq_stream_t stream) {
  if (!sh) return set_error(BQ_EINVAL, "bq_shard_check: shard is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int status = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&status, sh->dev.status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && status) e = cudaMemset(sh->dev.status, 0, sizeof(int));
  if (e != cudaSuccess) return set_error(BQ_ECUDA, std::string("bq_shard_check: ") + cudaGetErrorString(e));
  if (status)
    return set_error(BQ_ECUDA, "bq_step_adam8: device check " + std::to_string(status) +
                                   (status == 8 ? " (a tile region larger than 128x128)" : " (a wait timed out)"));
  return BQ_OK;
}

int bq_muon_ns_workspace(int batch, const bq_mat* mats, size_t* bytes) { return muon_ns_workspace(batch, mats, bytes); }

int bq_muon_ns(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps, void* ws,
               size_t ws_bytes, bq_stream_t stream) {
  return muon_ns(batch, mats, steps, a, b, c, eps, ws, ws_bytes, stream);
}

int bq_muon_ns_check(const void* ws, size_t ws_bytes, bq_stream_t stream) {
  return muon_ns_check(ws, ws_bytes, stream);
}

int bq_muon_ns_noalloc(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps,
                       bq_stream_t stream) {
  return muon_ns_noalloc(batch, mats, steps, a, b, c, eps, stream);
}

}  // extern "C"
