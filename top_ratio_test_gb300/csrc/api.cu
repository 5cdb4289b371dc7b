// C ABI of libserac_gb300: argument checks, image staging plan, workspace layout,
// the work schedule of the persistent fused kernel, and the launch sequence.
//
// Schedule.  Every pair is two row problems for the fused kernel: the rows of A
// against the columns B (its row top-2) and the rows of B against the columns A (its
// column top-2).  Pairs are processed in launch chunks of at most MAX_PAIRS pairs (the
// per-problem tables travel as kernel parameters, so a call needs no host-to-device
// copy and can be captured in a CUDA graph).  Within a chunk every problem's tiles are
// cut into as many pieces as there are persistent CTAs (fewer for small problems), one
// piece per CTA, with the CTA of a problem's first piece rotating from problem to
// problem so that the CTAs' tile counts stay within one tile per problem of each
// other; every CTA walks the problems in the same order, so the pairs in flight share
// L2.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <utility>
#include <vector>

#include "serac.h"
#include "serac_internal.h"

namespace serac {
namespace {

constexpr int64_t CHUNK_KEY_BYTES = 64ll << 20;
constexpr size_t ALIGN = 1024;

size_t align_up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

struct Chunk {
  int p0 = 0, p1 = 0;          // pairs [p0, p1)
  int img0 = 0, img1 = 0;      // images first used by this chunk: [img0, img1)
  int64_t tiles = 0;           // 128 x 256 tiles of all its problems (two per pair)
  int64_t rows = 0, cols = 0;  // sum of n_a, n_b
  int64_t blocks = 0;          // match-kernel blocks
};

struct Plan {
  std::vector<StageImage> images;  // unique images with their staged row offsets
  std::vector<int> a_img, b_img;   // per pair
  int64_t staged_rows = 0;
  std::vector<Chunk> chunks;
  size_t off_err = 0, off_staged = 0;
  // two chunk regions (chunk k uses region k % 2): keys, tickets, look-back status
  size_t off_region[2] = {0, 0}, region_bytes = 0, r_rowkeys = 0, r_colkeys = 0, r_tickets = 0, r_status = 0;
  size_t total = 0;
};

int64_t row_tiles(int32_t n_a) { return (static_cast<int64_t>(n_a) + BM - 1) / BM; }
int64_t col_tiles(int32_t n_b) { return (static_cast<int64_t>(n_b) + BN - 1) / BN; }

int64_t match_blocks(int32_t n_a) { return std::max<int64_t>(1, (static_cast<int64_t>(n_a) + MATCH_ROWS_PER_BLOCK - 1) / MATCH_ROWS_PER_BLOCK); }

// Tiles of the row problem of n_rows rows against n_cols columns.
int64_t problem_tiles(int32_t n_rows, int32_t n_cols) {
  if (n_rows <= 0 || n_cols <= 0) return 0;
  return row_tiles(n_rows) * col_tiles(n_cols);
}

// Tiles of a pair: its rows against B's descriptors, and B's rows against A's.
int64_t pair_tiles(const serac_pair& pr) { return problem_tiles(pr.n_a, pr.n_b) + problem_tiles(pr.n_b, pr.n_a); }

// Tiles of problem 2k (orientation 0: A's rows) or 2k + 1 (orientation 1: B's rows) of
// the pairs [p0, p1).
int64_t chunk_problem_tiles(const serac_pair* pairs, int p0, int problem) {
  const serac_pair& pr = pairs[p0 + problem / 2];
  return (problem & 1) ? problem_tiles(pr.n_b, pr.n_a) : problem_tiles(pr.n_a, pr.n_b);
}

void build_plan(const serac_pair* pairs, int32_t n_pairs, Plan& pl) {
  std::map<std::pair<const uint8_t*, int32_t>, int> seen;
  auto image_of = [&](const uint8_t* ptr, int32_t n) {
    auto key = std::make_pair(ptr, n);
    auto it = seen.find(key);
    if (it != seen.end()) return it->second;
    const int idx = static_cast<int>(pl.images.size());
    StageImage im;
    im.src = ptr;
    im.n = n;
    im.row0 = static_cast<int32_t>(pl.staged_rows);
    pl.staged_rows += round_up(n, PAD_ROWS);
    pl.images.push_back(im);
    seen.emplace(key, idx);
    return idx;
  };
  pl.a_img.resize(n_pairs);
  pl.b_img.resize(n_pairs);
  for (int p = 0; p < n_pairs; ++p) {
    pl.a_img[p] = image_of(pairs[p].a, pairs[p].n_a);
    pl.b_img[p] = image_of(pairs[p].b, pairs[p].n_b);
  }
  // chunks of consecutive pairs, bounded by the kernel-parameter tables and by the
  // key arrays (16 B per row and per column) they need
  int p = 0;
  while (p < n_pairs || (n_pairs == 0 && pl.chunks.empty())) {
    Chunk ch;
    ch.p0 = p;
    int64_t keys = 0;
    while (p < n_pairs && p - ch.p0 < MAX_PAIRS) {
      const int64_t kp = static_cast<int64_t>(pairs[p].n_a) + pairs[p].n_b;
      if (p > ch.p0 && (keys + kp) * 16 > CHUNK_KEY_BYTES) break;
      keys += kp;
      ++p;
    }
    ch.p1 = p;
    // images are numbered in order of first use, so each chunk's new ones are a range
    ch.img0 = pl.chunks.empty() ? 0 : pl.chunks.back().img1;
    ch.img1 = ch.img0;
    for (int k = ch.p0; k < ch.p1; ++k) {
      ch.img1 = std::max({ch.img1, pl.a_img[k] + 1, pl.b_img[k] + 1});
      ch.tiles += pair_tiles(pairs[k]);
      ch.rows += pairs[k].n_a;
      ch.cols += pairs[k].n_b;
      ch.blocks += match_blocks(pairs[k].n_a);
    }
    pl.chunks.push_back(ch);
    if (n_pairs == 0) break;
  }
  int64_t max_rows = 0, max_cols = 0, max_blocks = 0;
  for (const Chunk& ch : pl.chunks) {
    max_rows = std::max(max_rows, ch.rows);
    max_cols = std::max(max_cols, ch.cols);
    max_blocks = std::max(max_blocks, ch.blocks);
  }
  size_t off = 0;
  pl.off_err = off;
  off = align_up(off + 256);
  pl.off_staged = off;
  off = align_up(off + static_cast<size_t>(pl.staged_rows) * KDIM * 2);
  size_t r = 0;
  pl.r_rowkeys = r;
  r = align_up(r + static_cast<size_t>(max_rows) * 16);
  pl.r_colkeys = r;
  r = align_up(r + static_cast<size_t>(max_cols) * 16);
  pl.r_tickets = r;
  r = align_up(r + static_cast<size_t>(MAX_PAIRS) * 4);
  pl.r_status = r;
  r = align_up(r + static_cast<size_t>(max_blocks) * 8);
  pl.region_bytes = r;
  pl.off_region[0] = off;
  pl.off_region[1] = pl.chunks.size() > 1 ? off + r : off;  // one chunk needs one region
  off += pl.chunks.size() > 1 ? 2 * r : r;
  pl.total = off;
}

// CTAs of a chunk's launch: one per SM, at most one per tile.
int chunk_grid(const Chunk& ch, int sms) {
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({static_cast<int64_t>(sms), ch.tiles, MAX_GRID})));
}

// Tiles of piece k when T tiles are dealt to n pieces: T / n each, and one more for
// the first T mod n pieces.
int64_t piece_tiles(int64_t t, int n, int k) { return t / n + (k < t % n ? 1 : 0); }

// Column tiles of problem k of a chunk (a row tile's run of tiles).
int64_t chunk_problem_cols(const serac_pair* pairs, int p0, int problem) {
  const serac_pair& pr = pairs[p0 + problem / 2];
  return col_tiles((problem & 1) ? pr.n_a : pr.n_b);
}

// A segment start (the row tile's load, the pipeline refilling, the row's merge into
// the global keys) costs about half a tile of work; whole-row dealing is taken only
// when this cost model puts it more than 2 % ahead (the model is approximate, and the
// whole-row dealing spreads the CTAs' loads by up to a piece).
constexpr double SEGMENT_COST_TILES = 0.5;
constexpr double ROWS_MARGIN = 0.98;

// Pieces per problem and the CTA of each problem's first piece, for the 2 (p1 - p0)
// problems of a chunk.  Two dealings are costed (per CTA: its tiles plus
// SEGMENT_COST_TILES per segment; the chunk costs its busiest CTA):
//   * fine: every problem cut into min(grid, T) pieces, i.e. one per CTA for a large
//     problem; over a chunk the CTAs' tiles differ by at most one (the pieces with a
//     tile more go to the CTAs after those that took the previous problem's);
//   * rows: pieces of S tiles, S = the chunk's tiles over 4 per CTA but at most one
//     row tile's run of column tiles, so that a chunk with far more work than CTAs is
//     dealt in whole row tiles (one segment each, no row split over CTAs); consecutive
//     problems' pieces go round the CTAs.
// A single large pair costs the same both ways and stays fine, as do batches of mixed
// sizes; batches of equal pairs -- small ones (one-tile segments when dealt fine) most
// of all -- go rows.
void plan_pieces(const serac_pair* pairs, const Chunk& ch, int grid, int32_t* npieces, int32_t* offset) {
  const int nprob = 2 * (ch.p1 - ch.p0);
  std::vector<int64_t> t(nprob), c(nprob);
  for (int k = 0; k < nprob; ++k) {
    t[k] = chunk_problem_tiles(pairs, ch.p0, k);
    c[k] = chunk_problem_cols(pairs, ch.p0, k);
  }
  const int64_t s_cap = std::max<int64_t>(1, ch.tiles / (static_cast<int64_t>(grid) * 4));
  std::vector<double> load(grid);
  auto deal = [&](bool rows, int32_t* np, int32_t* off) {
    std::fill(load.begin(), load.end(), 0.0);
    int o = 0;
    for (int k = 0; k < nprob; ++k) {
      np[k] = 0;
      off[k] = o;
      if (t[k] == 0) continue;
      const int64_t s = rows ? std::max<int64_t>(1, std::min(c[k], s_cap)) : 1;
      const int n = static_cast<int>(std::min<int64_t>(grid, (t[k] + s - 1) / s));
      np[k] = n;
      const int64_t q = t[k] / n, r = t[k] % n;
      for (int i = 0; i < n; ++i) {
        const int64_t t0 = i * q + std::min<int64_t>(i, r), len = q + (i < r ? 1 : 0);
        const int64_t segs = (t0 % c[k] + len + c[k] - 1) / c[k];
        load[(o + i) % grid] += static_cast<double>(len) + SEGMENT_COST_TILES * static_cast<double>(segs);
      }
      o = static_cast<int>(n == grid ? (o + t[k] % grid) % grid : (o + n) % grid);
    }
    return *std::max_element(load.begin(), load.end());
  };
  const double fine = deal(false, npieces, offset);
  std::vector<int32_t> np_rows(nprob), off_rows(nprob);
  const double rows = deal(true, np_rows.data(), off_rows.data());
  if (rows < ROWS_MARGIN * fine)
    for (int k = 0; k < nprob; ++k) {
      npieces[k] = np_rows[k];
      offset[k] = off_rows[k];
    }
}

// ------------------------------------------------------------------ device state
struct DeviceInfo {
  bool init = false;
  int ok = 0;
  int sms = 0;
};
DeviceInfo g_dev[64];

int device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SERAC_ECUDA;
  if (dev < 0 || dev >= 64) return SERAC_EUNSUPPORTED;
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SERAC_ECUDA;
    d.ok = (major == 10 && minor == 3) ? 1 : 0;
    d.sms = n;
    d.init = true;
  }
  if (!d.ok) return SERAC_EUNSUPPORTED;
  *sms = d.sms;
  return SERAC_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// One tensor map over the whole staged buffer: [rows][128] bf16, box 64 x 128,
// 128-byte swizzle (the layout the MMA's shared-memory descriptors describe).
int encode_staged_map(CUtensorMap* map, void* staged, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return SERAC_EUNSUPPORTED;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(KDIM), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(KDIM) * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, staged, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SERAC_OK : SERAC_ECUDA;
}

// profiling events of the calling thread's calls (serac_set_profile_events)
thread_local cudaEvent_t g_ev_begin = nullptr, g_ev_end = nullptr;

// Per host thread and device: a side stream on which match_batch stages the images of
// its later launch chunks while the earlier chunks compute, and the events that order
// it (one for the call's start, one per staged chunk).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t start = nullptr;
  std::vector<cudaEvent_t> staged;
  ~SideStream() {  // at thread exit; errors (a runtime already shut down) are ignored
    for (cudaEvent_t e : staged) cudaEventDestroy(e);
    if (start) cudaEventDestroy(start);
    if (stream) cudaStreamDestroy(stream);
  }
};
constexpr int MAX_DEVICES = 64;
thread_local SideStream t_side[MAX_DEVICES];

int side_stream(size_t n_events, SideStream** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return SERAC_ECUDA;
  SideStream& s = t_side[dev];
  if (!s.stream && (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess ||
                    cudaEventCreateWithFlags(&s.start, cudaEventDisableTiming) != cudaSuccess))
    return SERAC_ECUDA;
  while (s.staged.size() < n_events) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return SERAC_ECUDA;
    s.staged.push_back(e);
  }
  *out = &s;
  return SERAC_OK;
}
thread_local bool g_inject_no_copies = false;  // consumed by this thread's next call
thread_local int g_last_launches = 0;    // per calling thread
thread_local int g_last_cuda_error = 0;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_pairs(const serac_pair* pairs, int32_t n_pairs) {
  if (n_pairs < 0 || (n_pairs > 0 && !pairs)) return SERAC_EINVAL;
  for (int p = 0; p < n_pairs; ++p) {
    const serac_pair& pr = pairs[p];
    if (pr.n_a < 0 || pr.n_b < 0 || pr.n_a > SERAC_MAX_N || pr.n_b > SERAC_MAX_N) return SERAC_EINVAL;
    if ((pr.n_a > 0 && (!pr.a || !aligned(pr.a, 16))) || (pr.n_b > 0 && (!pr.b || !aligned(pr.b, 16))))
      return SERAC_EINVAL;
  }
  return SERAC_OK;
}

int check_params(const serac_params* p) {
  if (!p) return SERAC_EINVAL;
  if (p->ratio_num_sq < 0 || p->ratio_den_sq <= 0 || p->max_features < 0) return SERAC_EINVAL;
  return SERAC_OK;
}

// Descriptors of an image of n that take part under the feature cap: the first K.
int32_t capped(const serac_params* p, int32_t n) {
  return (p->max_features > 0 && n > p->max_features) ? p->max_features : n;
}

int check_out(const serac_out* o, int32_t n_a, int32_t n_b) {
  if (!o || !o->count || !aligned(o->count, 4) || o->capacity < 0) return SERAC_EINVAL;
  if (o->capacity > 0 && (!o->matches || !aligned(o->matches, 8))) return SERAC_EINVAL;
  if (o->row_top2 && !aligned(o->row_top2, 16)) return SERAC_EINVAL;
  if (o->col_top2 && !aligned(o->col_top2, 16)) return SERAC_EINVAL;
  (void)n_a;
  (void)n_b;
  return SERAC_OK;
}

#define SERAC_TRY_CUDA(x)                              \
  do {                                                 \
    const cudaError_t e_ = (x);                        \
    if (e_ != cudaSuccess) {                           \
      g_last_cuda_error = static_cast<int>(e_);        \
      return SERAC_ECUDA;                              \
    }                                                  \
  } while (0)

// The whole sequence: staging, then per chunk fused -> match (or the score dump
// when `dump` is set).
int run(const serac_pair* pairs, int32_t n_pairs, const serac_params* params, const serac_out* outs,
        int32_t* dump, void* workspace, size_t ws_bytes, void* stream) {
  g_last_launches = 0;
  int sms = 0;
  int st = device_info(&sms);
  if (st != SERAC_OK) return st;
  Plan pl;
  build_plan(pairs, n_pairs, pl);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < pl.total) return SERAC_EWORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* err = reinterpret_cast<int32_t*>(ws + pl.off_err);
  uint16_t* staged = reinterpret_cast<uint16_t*>(ws + pl.off_staged);

  CUtensorMap map;
  if (pl.staged_rows > 0) {
    st = encode_staged_map(&map, staged, pl.staged_rows);
    if (st != SERAC_OK) return st;
  }

  // staging, one launch per chunk for the images it uses first (at most 256).  The
  // first launch also clears the error word and the key arrays, which every match
  // launch leaves cleared behind it.  With several chunks, the later chunks' images
  // are staged on a side stream while the earlier chunks compute (their host reads
  // overlap the kernels); each chunk's fused launch waits for its own staging.
  const bool overlap = pl.chunks.size() > 1 && !dump;
  SideStream* side = nullptr;
  std::vector<char> on_side(pl.chunks.size(), 0);  // chunk staged on the side stream
  if (overlap) {
    st = side_stream(pl.chunks.size(), &side);
    if (st != SERAC_OK) return st;
  }
  for (size_t ci = 0; ci < pl.chunks.size(); ++ci) {
    const Chunk& ch = pl.chunks[ci];
    StageParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.staged = staged;
    sp.err = err;
    if (ci == 0) {
      sp.zero = reinterpret_cast<uint4*>(ws + pl.off_region[0]);
      sp.zero_n = static_cast<int64_t>((pl.total - pl.off_region[0]) / 16);
      sp.zero_blocks = static_cast<int32_t>(std::min<int64_t>(1024, (sp.zero_n + 255) / 256));
      if (sp.zero_blocks < 1) sp.zero_blocks = 1;
    }
    int64_t max_chunks = 0;
    for (int i = ch.img0; i < ch.img1; ++i) {
      if (pl.images[i].n == 0) continue;
      sp.images[sp.n_images++] = pl.images[i];
      max_chunks = std::max<int64_t>(max_chunks, round_up(pl.images[i].n, PAD_ROWS) * (KDIM / 16));
    }
    if (ci > 0 && sp.n_images == 0) continue;
    void* s_stage = (ci == 0 || !overlap) ? stream : static_cast<void*>(side->stream);
    SERAC_TRY_CUDA(static_cast<cudaError_t>(launch_stage(sp, max_chunks, s_stage, s_stage != stream)));
    ++g_last_launches;
    if (ci == 0 && overlap) {
      // the side stream starts once the first chunk is staged: it then has the host
      // link to itself while the first chunk computes, and the work queued earlier on
      // `stream` (a previous call with this workspace) is done
      SERAC_TRY_CUDA(cudaEventRecord(side->start, static_cast<cudaStream_t>(stream)));
      SERAC_TRY_CUDA(cudaStreamWaitEvent(side->stream, side->start, 0));
    }
    if (ci > 0 && overlap) {
      SERAC_TRY_CUDA(cudaEventRecord(side->staged[ci], side->stream));
      on_side[ci] = 1;
    }
  }

  bool first_fused = true;
  for (size_t ci = 0; ci < pl.chunks.size(); ++ci) {
    const Chunk& ch = pl.chunks[ci];
    uint8_t* region = ws + pl.off_region[ci & 1];
    uint8_t* other = ws + pl.off_region[(ci + 1) & 1];
    unsigned long long* rowkeys = reinterpret_cast<unsigned long long*>(region + pl.r_rowkeys);
    unsigned long long* colkeys = reinterpret_cast<unsigned long long*>(region + pl.r_colkeys);
    // this chunk's images (staged on the side stream) must be in place
    if (on_side[ci]) SERAC_TRY_CUDA(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), side->staged[ci], 0));
    // ---------------- fused GEMM + row top-2 of both problems of every pair
    if (ch.tiles > 0) {
      FusedParams fp;
      std::memset(&fp, 0, sizeof(fp));
      fp.grid = chunk_grid(ch, sms);
      int32_t npieces[MAX_PROBLEMS], offset[MAX_PROBLEMS];
      plan_pieces(pairs, ch, fp.grid, npieces, offset);
      fp.err = err;
      fp.dump = dump;
      fp.dump_ld = (dump && n_pairs > 0) ? pairs[0].n_b : 0;
      fp.key_mult = 256u;
      // the last chunk's match grid, if it has at most one block per SM, may start
      // beside the fused CTAs (its blocks fit there) and wait for them
      int64_t mblocks = 0;
      for (int k = ch.p0; k < ch.p1; ++k) mblocks += match_blocks(pairs[k].n_a);
      fp.early_dependents = (!dump && ci + 1 == pl.chunks.size() && mblocks <= sms) ? 1 : 0;
      fp.no_copies = (first_fused && g_inject_no_copies) ? 1 : 0;
      if (first_fused) g_inject_no_copies = false;
      int np = 0;
      int64_t rows = 0, cols = 0;
      for (int k = ch.p0; k < ch.p1; ++k) {
        const int32_t ra = pl.images[pl.a_img[k]].row0, rb = pl.images[pl.b_img[k]].row0;
        for (int o = 0; o < 2; ++o) {
          const int pi = 2 * (k - ch.p0) + o;
          if (npieces[pi] == 0) continue;
          FusedPair& f = fp.pairs[np++];
          f.a_row0 = o ? rb : ra;
          f.b_row0 = o ? ra : rb;
          f.n_a = o ? pairs[k].n_b : pairs[k].n_a;
          f.n_b = o ? pairs[k].n_a : pairs[k].n_b;
          f.npieces = npieces[pi];
          f.offset = offset[pi];
          f.transposed = o;
          f.keys = o ? colkeys + 2 * cols : rowkeys + 2 * rows;
        }
        rows += pairs[k].n_a;
        cols += pairs[k].n_b;
      }
      fp.n_pairs = np;
      const bool prof = first_fused && g_ev_begin && g_ev_end;
      if (prof)
        SERAC_TRY_CUDA(cudaEventRecordWithFlags(g_ev_begin, static_cast<cudaStream_t>(stream), cudaEventRecordExternal));
      SERAC_TRY_CUDA(static_cast<cudaError_t>(launch_fused(fp, &map, dump ? MODE_DUMP : MODE_TOP2, stream)));
      ++g_last_launches;
      if (prof)
        SERAC_TRY_CUDA(cudaEventRecordWithFlags(g_ev_end, static_cast<cudaStream_t>(stream), cudaEventRecordExternal));
      first_fused = false;
    }
    if (dump) continue;
    // ---------------- decisions and compaction (clears the keys it read)
    FinishParams fn;
    std::memset(&fn, 0, sizeof(fn));
    fn.ratio_num_sq = params->ratio_num_sq;
    fn.ratio_den_sq = params->ratio_den_sq;
    fn.norm_sq = params->norm_sq;
    fn.min_score = params->min_score;
    fn.mutual = params->mutual;
    fn.col_ratio = params->col_ratio;
    fn.rowkeys = rowkeys;
    fn.colkeys = colkeys;
    fn.tickets = reinterpret_cast<int32_t*>(region + pl.r_tickets);
    fn.status = reinterpret_cast<unsigned long long*>(region + pl.r_status);
    // the next chunk's region was last used by the previous chunk, whose match
    // launch has finished before this chunk's fused launch began
    fn.zero = pl.chunks.size() > 1 ? reinterpret_cast<uint4*>(other) : nullptr;
    fn.zero_n = pl.chunks.size() > 1 ? static_cast<int64_t>(pl.region_bytes / 16) : 0;
    fn.err = err;
    int64_t rows = 0, cols = 0, blocks = 0;
    int np = 0;
    for (int k = ch.p0; k < ch.p1; ++k) {
      FinishPair& f = fn.pairs[np++];
      f.n_a = pairs[k].n_a;
      f.n_b = pairs[k].n_b;
      f.row_base = static_cast<int32_t>(rows);
      f.col_base = static_cast<int32_t>(cols);
      f.matches = outs[k].matches;
      f.count = outs[k].count;
      f.row_top2 = outs[k].row_top2;
      f.col_top2 = outs[k].col_top2;
      f.capacity = outs[k].capacity;
      f.blk_base = static_cast<int32_t>(blocks);
      f.nblk = static_cast<int32_t>(match_blocks(pairs[k].n_a));
      blocks += f.nblk;
      rows += pairs[k].n_a;
      cols += pairs[k].n_b;
    }
    fn.n_pairs = np;
    fn.total_blocks = static_cast<int32_t>(blocks);
    if (np > 0) {
      SERAC_TRY_CUDA(static_cast<cudaError_t>(launch_match(fn, stream)));
      ++g_last_launches;
    }
  }
  return SERAC_OK;
}

// ------------------------------------------------------------------ row top-k
// One row problem (A's rows against B) on the persistent fused kernel in a top-k mode,
// then the merge of its segment lists.  Workspace: the error word, A and B staged as
// bf16, the lists (slots x 4 quarters x K keys per row, slots = the most pieces that
// cover one row tile).
struct TopkPlan {
  int K = 4, grid = 1, npieces = 1, slots = 0, ldl = 0;
  int64_t tiles = 0;
  size_t off_err = 0, off_staged = 0, off_lists = 0, total = 0;
  int64_t staged_rows = 0;
};

int topk_plan(int32_t n_a, int32_t n_b, int32_t k, int sms, TopkPlan& tp) {
  if (k < 1 || k > MAX_TOPK || n_a < 0 || n_b < 0 || n_a > SERAC_MAX_N || n_b > SERAC_MAX_N) return SERAC_EINVAL;
  tp.K = k <= 4 ? MODE_TOPK4 : MODE_TOPK8;
  tp.tiles = problem_tiles(n_a, n_b);
  tp.grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({static_cast<int64_t>(sms), tp.tiles, MAX_GRID})));
  tp.npieces = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tp.grid, tp.tiles)));
  tp.ldl = static_cast<int>(round_up(std::max(n_a, 1), BM));
  tp.slots = 0;
  const int64_t ct = col_tiles(n_b);
  for (int64_t rt = 0; tp.tiles > 0 && rt < row_tiles(n_a); ++rt) {
    const int64_t t0 = rt * ct, t1 = std::min(tp.tiles, t0 + ct);
    tp.slots = std::max(tp.slots, piece_of(t1 - 1, tp.tiles, tp.npieces) - piece_of(t0, tp.tiles, tp.npieces) + 1);
  }
  tp.staged_rows = round_up(n_a, PAD_ROWS) + round_up(n_b, PAD_ROWS);
  size_t off = 0;
  tp.off_err = off;
  off = align_up(off + 256);
  tp.off_staged = off;
  off = align_up(off + static_cast<size_t>(tp.staged_rows) * KDIM * 2);
  tp.off_lists = off;
  off = align_up(off + static_cast<size_t>(tp.slots) * 4 * tp.K * tp.ldl * 8);
  tp.total = off;
  return SERAC_OK;
}

static_assert(MAX_TOPK == SERAC_MAX_TOPK, "one top-k limit");

int run_topk(const uint8_t* a, int32_t n_a, const uint8_t* b, int32_t n_b, int32_t k, int32_t* scores,
             int32_t* index, int32_t* status, void* workspace, size_t ws_bytes, void* stream) {
  g_last_launches = 0;
  int sms = 0;
  int st = device_info(&sms);
  if (st != SERAC_OK) return st;
  TopkPlan tp;
  st = topk_plan(n_a, n_b, k, sms, tp);
  if (st != SERAC_OK) return st;
  if (!workspace || !aligned(workspace, 256) || ws_bytes < tp.total) return SERAC_EWORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* err = reinterpret_cast<int32_t*>(ws + tp.off_err);
  uint16_t* staged = reinterpret_cast<uint16_t*>(ws + tp.off_staged);
  CUtensorMap map;
  st = encode_staged_map(&map, staged, tp.staged_rows);
  if (st != SERAC_OK) return st;
  // staging (clears the error word); the lists need no clearing: the merge reads only
  // the slots the row's segments write
  StageParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.staged = staged;
  sp.err = err;
  sp.zero_blocks = 1;  // its first block clears the error word (nothing else to clear)
  int64_t max_chunks = 0;
  const int32_t b_row0 = static_cast<int32_t>(round_up(n_a, PAD_ROWS));
  if (n_a > 0) sp.images[sp.n_images++] = StageImage{a, n_a, 0};
  if (n_b > 0) sp.images[sp.n_images++] = StageImage{b, n_b, b_row0};
  for (int i = 0; i < sp.n_images; ++i)
    max_chunks = std::max<int64_t>(max_chunks, round_up(sp.images[i].n, PAD_ROWS) * (KDIM / 16));
  SERAC_TRY_CUDA(static_cast<cudaError_t>(launch_stage(sp, max_chunks, stream, false)));
  ++g_last_launches;
  unsigned long long* lists = reinterpret_cast<unsigned long long*>(ws + tp.off_lists);
  if (tp.tiles > 0) {
    FusedParams fp;
    std::memset(&fp, 0, sizeof(fp));
    fp.grid = tp.grid;
    fp.err = err;
    fp.key_mult = 256u;
    fp.no_copies = g_inject_no_copies ? 1 : 0;
    g_inject_no_copies = false;
    FusedPair& f = fp.pairs[0];
    f.a_row0 = 0;
    f.b_row0 = b_row0;
    f.n_a = n_a;
    f.n_b = n_b;
    f.npieces = tp.npieces;
    f.offset = 0;
    f.ldl = tp.ldl;
    f.keys = lists;
    fp.n_pairs = 1;
    const bool prof = g_ev_begin && g_ev_end;
    if (prof)
      SERAC_TRY_CUDA(cudaEventRecordWithFlags(g_ev_begin, static_cast<cudaStream_t>(stream), cudaEventRecordExternal));
    SERAC_TRY_CUDA(static_cast<cudaError_t>(launch_fused(fp, &map, tp.K, stream)));
    ++g_last_launches;
    if (prof)
      SERAC_TRY_CUDA(cudaEventRecordWithFlags(g_ev_end, static_cast<cudaStream_t>(stream), cudaEventRecordExternal));
  }
  TopkMergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.lists = lists;
  mp.n_a = n_a;
  mp.n_b = n_b;
  mp.ldl = tp.ldl;
  mp.npieces = tp.npieces;
  mp.k = k;
  mp.scores = scores;
  mp.index = index;
  mp.status = status;
  mp.err = err;
  SERAC_TRY_CUDA(static_cast<cudaError_t>(launch_topk_merge(mp, tp.K, stream)));
  ++g_last_launches;
  return SERAC_OK;
}

}  // namespace
}  // namespace serac

using namespace serac;

extern "C" {

int serac_default_params(serac_params* p, float max_ratio, float max_angle_rad) {
  if (!p || !(max_ratio > 0.0f) || max_ratio > 1.0f || !(max_angle_rad >= 0.0f) ||
      max_angle_rad > 1.5707964f)
    return SERAC_EINVAL;
  const int64_t r = static_cast<int64_t>(std::llround(static_cast<double>(max_ratio) * 10000.0));
  int64_t num = r * r, den = 100000000;
  int64_t a = num, b = den;
  while (b) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  num /= a;
  den /= a;
  const int32_t n = 512 * 512;
  p->ratio_num_sq = static_cast<int32_t>(num);
  p->ratio_den_sq = static_cast<int32_t>(den);
  p->norm_sq = n;
  p->min_score = static_cast<int32_t>(std::ceil(std::cos(static_cast<double>(max_angle_rad)) * n));
  p->mutual = 1;
  p->col_ratio = 1;
  p->max_features = 0;
  return SERAC_OK;
}

size_t serac_pair_workspace_size(int32_t n_a, int32_t n_b) {
  serac_pair pr;
  pr.a = reinterpret_cast<const uint8_t*>(16);
  pr.b = reinterpret_cast<const uint8_t*>(32);
  pr.n_a = n_a < 0 ? 0 : n_a;
  pr.n_b = n_b < 0 ? 0 : n_b;
  Plan pl;
  build_plan(&pr, 1, pl);
  return pl.total;
}

size_t match_batch_workspace_size(const serac_pair* pairs, int32_t n_pairs) {
  if (check_pairs(pairs, n_pairs) != SERAC_OK) return 0;
  Plan pl;
  build_plan(pairs, n_pairs, pl);
  return pl.total;
}

int match_pair(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b,
               const serac_params* params, const serac_out* out, void* workspace, size_t workspace_bytes,
               void* cuda_stream) {
  serac_pair pr;
  pr.a = desc_a;
  pr.n_a = n_a;
  pr.b = desc_b;
  pr.n_b = n_b;
  int st = check_pairs(&pr, 1);
  if (st == SERAC_OK) st = check_params(params);
  if (st == SERAC_OK) st = check_out(out, n_a, n_b);
  if (st != SERAC_OK) return st;
  pr.n_a = capped(params, n_a);
  pr.n_b = capped(params, n_b);
  return run(&pr, 1, params, out, nullptr, workspace, workspace_bytes, cuda_stream);
}

int match_batch(const serac_pair* pairs, int32_t n_pairs, const serac_params* params, const serac_out* outs,
                void* workspace, size_t workspace_bytes, void* cuda_stream) {
  int st = check_pairs(pairs, n_pairs);
  if (st == SERAC_OK) st = check_params(params);
  if (st != SERAC_OK) return st;
  if (n_pairs > 0 && !outs) return SERAC_EINVAL;
  for (int p = 0; p < n_pairs; ++p) {
    st = check_out(&outs[p], pairs[p].n_a, pairs[p].n_b);
    if (st != SERAC_OK) return st;
  }
  if (params->max_features == 0)
    return run(pairs, n_pairs, params, outs, nullptr, workspace, workspace_bytes, cuda_stream);
  std::vector<serac_pair> cp(pairs, pairs + n_pairs);
  for (serac_pair& pr : cp) {
    pr.n_a = capped(params, pr.n_a);
    pr.n_b = capped(params, pr.n_b);
  }
  return run(cp.data(), n_pairs, params, outs, nullptr, workspace, workspace_bytes, cuda_stream);
}

int serac_scores(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b, int32_t* scores,
                 void* workspace, size_t workspace_bytes, void* cuda_stream) {
  serac_pair pr;
  pr.a = desc_a;
  pr.n_a = n_a;
  pr.b = desc_b;
  pr.n_b = n_b;
  int st = check_pairs(&pr, 1);
  if (st != SERAC_OK) return st;
  if (static_cast<int64_t>(n_a) * n_b > 0 && (!scores || !aligned(scores, 4))) return SERAC_EINVAL;
  serac_params dummy;
  serac_default_params(&dummy, 0.8f, 0.7f);
  return run(&pr, 1, &dummy, nullptr, scores ? scores : reinterpret_cast<int32_t*>(16), workspace,
             workspace_bytes, cuda_stream);
}

size_t serac_topk_workspace_size(int32_t n_a, int32_t n_b, int32_t k) {
  int sms = 0;
  if (device_info(&sms) != SERAC_OK) return 0;
  TopkPlan tp;
  if (topk_plan(n_a, n_b, k, sms, tp) != SERAC_OK) return 0;
  return tp.total;
}

int serac_topk_pair(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b, int32_t k,
                    int32_t* scores, int32_t* index, int32_t* status, void* workspace, size_t workspace_bytes,
                    void* cuda_stream) {
  serac_pair pr;
  pr.a = desc_a;
  pr.n_a = n_a;
  pr.b = desc_b;
  pr.n_b = n_b;
  int st = check_pairs(&pr, 1);
  if (st != SERAC_OK) return st;
  if (k < 1 || k > SERAC_MAX_TOPK) return SERAC_EINVAL;
  if (n_a > 0 && (!scores || !index || !aligned(scores, 4) || !aligned(index, 4))) return SERAC_EINVAL;
  if (status && !aligned(status, 4)) return SERAC_EINVAL;
  return run_topk(desc_a, n_a, desc_b, n_b, k, scores, index, status, workspace, workspace_bytes, cuda_stream);
}

int serac_set_profile_events(void* ev_begin, void* ev_end) {
  g_ev_begin = static_cast<cudaEvent_t>(ev_begin);
  g_ev_end = static_cast<cudaEvent_t>(ev_end);
  return SERAC_OK;
}

int serac_test_inject_timeout(int enable) {
  g_inject_no_copies = enable != 0;
  return SERAC_OK;
}

int serac_device_check(void) {
  int sms = 0;
  return device_info(&sms);
}

int serac_last_launch_count(void) { return g_last_launches; }

int serac_last_cuda_error(void) { return g_last_cuda_error; }

int serac_schedule_describe(const serac_pair* pairs, int32_t n_pairs, int32_t grid, int32_t* out_chunks,
                            int32_t* out_pieces, int32_t* out_npieces, int32_t* cta_tiles) {
  if (check_pairs(pairs, n_pairs) != SERAC_OK || grid <= 0 || grid > MAX_GRID) return SERAC_EINVAL;
  Plan pl;
  build_plan(pairs, n_pairs, pl);
  if (out_chunks) *out_chunks = static_cast<int32_t>(pl.chunks.size());
  const Chunk& ch = pl.chunks.front();
  const int g = chunk_grid(ch, grid);
  int32_t npieces[MAX_PROBLEMS], offset[MAX_PROBLEMS];
  plan_pieces(pairs, ch, g, npieces, offset);
  const int nprob = 2 * (ch.p1 - ch.p0);
  int64_t total = 0;
  for (int k = 0; k < nprob; ++k) total += npieces[k];
  if (out_pieces) *out_pieces = static_cast<int32_t>(total);
  if (out_npieces)
    for (int k = 0; k < nprob; ++k) out_npieces[k] = npieces[k];
  if (cta_tiles) {
    for (int c = 0; c < grid; ++c) cta_tiles[c] = 0;
    for (int k = 0; k < nprob; ++k) {
      const int64_t t = chunk_problem_tiles(pairs, ch.p0, k);
      for (int i = 0; i < npieces[k]; ++i)
        cta_tiles[(offset[k] + i) % g] += static_cast<int32_t>(piece_tiles(t, npieces[k], i));
    }
  }
  return SERAC_OK;
}

const char* serac_status_str(int status) {
  switch (status) {
    case SERAC_OK: return "ok";
    case SERAC_EINVAL: return "invalid argument";
    case SERAC_ECAPACITY: return "match buffer too small (count holds the needed size)";
    case SERAC_ECUDA: return "CUDA runtime error";
    case SERAC_ETIMEOUT: return "a bounded wait inside a kernel ran out";
    case SERAC_EWORKSPACE: return "workspace missing, misaligned or too small";
    case SERAC_EUNSUPPORTED: return "device is not sm_103 or TMA encoding is unavailable";
    default: return "unknown status";
  }
}

}  // extern "C"
