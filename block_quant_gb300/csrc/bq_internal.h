// Internal structures shared by the host side of libbq (planner, work-table
// builder, C ABI) and the step kernels.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/bq.h"

namespace bq {

// ---------------------------------------------------------------- layout (host)

struct Tensor {
  int64_t rows, cols, g, numel;
  int32_t adam_kind, fp8;
  bool one_d() const { return rows == 1; }
  // elements of one 128-row band of the 2-D view (1-D: one 1x128 tile)
  int64_t band() const { return one_d() ? 128 : 128 * cols; }
};

struct Interval {
  int64_t dev, tensor, t_off, len, local_off, mslot, fslot;
};

}  // namespace bq

struct bq_layout {
  int64_t V = 0, S = 0, alpha = 0, start_align = 0, case3 = 0;
  std::vector<bq::Tensor> tensors;
  std::vector<int64_t> start;
  std::vector<bq::Interval> intervals;
  std::vector<int64_t> dev_first, dev_mslot, dev_fslot;  // V + 1 entries each
  int64_t n_mslots = 0, n_fslots = 0;
};

namespace bq {

// ---------------------------------------------------------------- device work tables

// pack: the destination range of a shard split into chunks of kPackChunk
// elements; every chunk is covered by consecutive pieces that never cross a
// chunk boundary.  tensor < 0 marks padding (written as +0).
constexpr int64_t kPackChunk = 16384;
struct PackPiece {
  int64_t dst;     // local element position
  int64_t src;     // tensor-flat element offset
  int32_t len;     // elements
  int32_t tensor;  // index into grad_ptrs, -1 = padding
};

// A run of whole flat Adam blocks of one tensor (blocks of 256 or 128
// elements from pos; the last one may be short).  fslot >= 0: the tensor is
// 1-D with FP8 1x128 tiles, numbered from fslot in flat order.
struct FlatGroup {
  int64_t pos;
  int32_t nelem;
  int32_t mslot;
  int32_t fslot;
  int32_t pad_;
};

// A rectangular region of a 2-D tensor: rows x [c0, c0 + width) with row pitch C,
// pos = local position of (row 0, column c0).  Used for
//  - FLAT256 Adam + FP8 (strip): width == C (whole band, flat 256-element
//    blocks over rows*C from pos) or, when C % 256 == 0, a multiple of 256
//    columns (blocks are 256-column row segments, block (r, j) has slot
//    mslot + r*(C/256) + j); FP8 tile t = columns c0 + 128t, slot fslot + t.
//  - TILE128 Adam (tile): width <= 128, one tile, Adam slot mslot, FP8 slot fslot.
//  A 256-column strip also names its interval's 2-D tensor maps: tm (-1: none)
//  and trow, the strip's first row within that interval.
struct RegionGroup {
  int64_t pos;
  int32_t rows, C, c0, width;
  int32_t mslot, fslot;
  uint32_t cmul, cshr;  // n / C == umulhi(n, cmul) >> cshr for 0 <= n < 2^31 (cmul 0: C == 1)
  int32_t tm = -1, trow = 0;
};

// The rows [0, rows) x C of one 2-D tensor interval that strips cover, from local
// position pos: the strip kernel reads them through four 2-D tensor maps (grad,
// master, m, v) built for the caller's buffers, 8 rows x 256 columns a copy.
struct MapInterval {
  int64_t pos;
  int32_t C, rows;
};
constexpr int kMapBytes = 128;  // one CUtensorMap

// Division by an invariant integer with a multiply and a shift (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994):
// with l = ceil(log2 d) and m = ceil(2^(31+l) / d), floor(n / d) equals
// floor(n * m / 2^(31+l)) for every 0 <= n < 2^31.
inline void make_fastdiv(uint32_t d, uint32_t* mul, uint32_t* shr) {
  if (d <= 1) {
    *mul = 0;
    *shr = 0;
    return;
  }
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  *mul = uint32_t(((uint64_t(1) << (31 + l)) + d - 1) / d);
  *shr = l - 1;
}

struct ShardTables {
  std::vector<PackPiece> pieces;
  std::vector<int32_t> chunk_first;   // nchunks + 1
  std::vector<FlatGroup> flat256;     // FLAT256 Adam blocks without 2-D FP8 tiles
  std::vector<FlatGroup> flat128;     // TILE128 Adam on 1-D tensors (128-element tiles)
  std::vector<RegionGroup> strips;    // FLAT256 Adam + 2-D FP8
  std::vector<RegionGroup> tiles;     // TILE128 Adam on 2-D tensors
  std::vector<PackPiece> muon;        // Muon tensors: dst local, src tensor offset, <= 8192 elements
  std::vector<FlatGroup> flat32;      // TILE32 Adam on 1-D tensors (32-element blocks)
  std::vector<RegionGroup> tiles32;   // TILE32 Adam on 2-D tensors: 32-row band x <= 256 columns
  std::vector<RegionGroup> band_tiles;  // FP8 tiles of FLAT256 tensors with C % 256 != 0 (one group each)
  std::vector<MapInterval> maps;        // the strips' tensor intervals (4 tensor maps each at step time)
  int64_t nchunks = 0;
  int32_t max_strip_tiles = 0;        // most FP8 column tiles in one strip group
};

void build_shard_tables(const bq_layout& L, int dev_lo, int dev_hi, ShardTables& T);
std::string validate_shard_tables(const bq_layout& L, int dev_lo, int dev_hi, const ShardTables& T);

// where one member of a group lives in the group's buffers and pointer arrays
struct GroupPlace {
  int64_t elem, mslot, fslot, tensor;
};
void append_member_tables(const ShardTables& member, const GroupPlace& at, ShardTables& group);
void finish_group_tables(int64_t group_total, ShardTables& group);

// ---------------------------------------------------------------- kernel launchers (step_kernels.cu)

struct DevTables {
  const PackPiece* pieces;
  const int32_t* chunk_first;
  const FlatGroup* flat256;
  const FlatGroup* flat128;
  const RegionGroup* strips;
  const RegionGroup* tiles;
  const PackPiece* muon;
  const FlatGroup* flat32;
  const RegionGroup* tiles32;
  const RegionGroup* band_tiles;
  int64_t nchunks;
  int32_t n_flat256, n_flat128, n_strips, n_tiles, n_muon, n_flat32, n_tiles32, n_band_tiles;
  int32_t max_strip_tiles;
  int* status;  // device error word: 0, or the site of a wait that timed out
  void* tmaps;  // 4 tensor maps (grad, master, m, v) per map interval, written before a step uses them
  int32_t n_maps;
};

struct AdamArgs {
  const uint16_t* grad;
  float* master;
  int8_t* m;
  uint8_t* v;
  float* m_scale;
  float* v_scale;
  uint8_t* fp8;      // may be null
  float* fp8_scale;  // may be null
  bq_adam_hp hp;
  int* status;          // device error word of the shard (set by the launcher)
  const void* tmaps;    // the strips' tensor maps for these buffers, or NULL (per-block copies)
};

int launch_pack(const DevTables& t, const uint16_t* const* grads, uint16_t* dst, int64_t total, float scale,
                int accumulate, void* stream);
int launch_adam8(const DevTables& t, const AdamArgs& a, void* stream);
int launch_quant_fp8(const DevTables& t, const float* master, uint8_t* fp8, float* fp8_scale, void* stream);
int launch_wait_selftest(int* status, void* stream);
int launch_dequant_fp8(const DevTables& t, const uint8_t* fp8, const float* fp8_scale, uint16_t* out, void* stream);
int launch_muon_momentum(const DevTables& t, const uint16_t* grad, float* mom, float mu, uint16_t* const* gather,
                         void* stream);
int launch_muon_apply(const DevTables& t, float* master, const uint16_t* const* upd, const float* lr, void* stream);

// Muon (ns_gemm.cu)
int muon_ns_workspace(int batch, const bq_mat* mats, size_t* bytes);
int muon_ns(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps, void* ws,
            size_t ws_bytes, void* stream);
int muon_ns_check(const void* ws, size_t ws_bytes, void* stream);
int muon_ns_noalloc(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps, void* stream);
// a 2-D tiled tensor map (no swizzle) over `rows` x `cols` elements of elem_bytes
// each at base with row pitch cols; boxes of box_cols x box_rows.  map: 128 bytes.
int encode_map_2d(void* map, const void* base, int elem_bytes, int64_t cols, int64_t rows, int box_cols, int box_rows);

// errors
int set_error(int code, const std::string& msg);
int sm_count();  // SMs of the current device (cached per device)
bool once_per_device(int key);  // true once per (current device, key); keys below
constexpr int kOnceStripAttr = 0, kOnceGemmAttr = 1, kOnceTileAttr = 2;

}  // namespace bq
