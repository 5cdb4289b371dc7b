// Internal layout shared by the host scheduler (api.cu) and the kernels.
//
// Both directions of a pair are row problems.  The column top-2 of the pair (A, B) is
// the row top-2 of (B, A), so every pair is matched as two problems of the same kind:
// rows of A against the columns B, and rows of B against the columns A.  The fused
// kernel only ever keeps row top-2s.
//
// Tiling: a problem's score matrix is cut into tiles of BM = 128 rows (one tcgen05
// accumulator: TMEM lane = row) by BN = 256 columns (TMEM columns).  Every image is
// staged once as bf16, zero-padded to a multiple of 256 rows, into one buffer that a
// single TMA tensor map covers; the zero rows score 0 and the zero floor drops them,
// so ragged tails need no masking.
//
// Work: in a launch chunk, every problem's T tiles are cut into n <= grid pieces (T / n
// tiles each, one more for the first T mod n); piece k of problem p goes to CTA
// (offset_p + k) mod grid of the persistent fused kernel.  A single large pair is cut
// into one piece per CTA; in a chunk with much more work than CTAs the pieces grow to
// whole row tiles (see plan_pieces).  A piece is a
// run of the problem's tiles in row-major order, processed as segments: one row tile
// resident in shared memory against a run of column tiles, with one running top-2 per
// row.  All CTAs thus work through the problems in the same order (a pair's two
// problems one after the other), so the operands in flight stay in L2, and every CTA
// gets the same number of tiles within one per problem.
#pragma once
#include <stdint.h>

namespace serac {

constexpr int BM = 128;          // rows of A per tile (MMA M, TMEM lanes)
constexpr int BN = 256;          // rows of B per tile (MMA N, TMEM columns)
constexpr int KDIM = 128;        // descriptor length
constexpr int PAD_ROWS = 256;    // staged images are padded to this many rows
constexpr int MAX_PAIRS = 128;   // pairs per launch (kernel-parameter tables)
constexpr int MAX_GRID = 256;    // persistent CTAs per launch
constexpr int FUSED_THREADS = 576;  // warp 0 TMA, warp 1 MMA, warps 2..17 epilogue

__host__ __device__ inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// error bits set by kernels (workspace word 0)
constexpr int ERR_TIMEOUT_PRODUCER = 1;
constexpr int ERR_TIMEOUT_MMA = 2;
constexpr int ERR_TIMEOUT_EPILOGUE = 4;
constexpr int ERR_TIMEOUT_LOOKBACK = 8;

// One row problem: rows of one staged image against the rows (columns of the score
// matrix) of another.
struct FusedPair {
  int32_t a_row0;      // first staged row of the row-side image
  int32_t b_row0;      // first staged row of the column-side image
  int32_t n_a, n_b;    // rows, columns
  int32_t npieces;     // pieces the problem's tiles are cut into (<= grid)
  int32_t offset;      // piece k goes to CTA (offset + k) mod grid
  int32_t transposed;  // score dump only: rows are the pair's B (write S[col][row])
  int32_t ldl;         // row top-k only: row stride of the segment lists (n_a rounded up to BM)
  unsigned long long* keys;  // [n_a][2] row keys of this problem (rowkeys or colkeys of the pair);
                             // row top-k: the segment lists (see topk_list_index)
};

// Epilogue modes of the fused kernel.
constexpr int MODE_TOP2 = 0;   // row top-2 of every problem, merged into the global keys
constexpr int MODE_DUMP = 1;   // the score matrix itself (small pairs, tests only)
constexpr int MODE_TOPK4 = 4;  // row top-4 per segment, written to segment lists
constexpr int MODE_TOPK8 = 8;  // row top-8 per segment, written to segment lists
constexpr int MAX_TOPK = 8;

// The piece that holds tile t when T tiles are dealt to n pieces (T / n tiles per piece
// and one more for the first T mod n pieces).
__host__ __device__ inline int32_t piece_of(int64_t t, int64_t T, int32_t n) {
  const int64_t q = T / n, r = T % n;
  if (t < r * (q + 1)) return static_cast<int32_t>(t / (q + 1));
  return static_cast<int32_t>(r + (t - r * (q + 1)) / q);
}

// Row top-k lists.  Every segment of a row problem (one piece's run of column tiles on
// one row tile) writes, per row and per 64-column quarter of the tiles, the K best
// 64-bit keys it saw, in descending order.  The segments of row tile rt are the
// pieces piece_of(rt C) .. piece_of(min(T, (rt + 1) C) - 1), C = column tiles; the
// piece's position in that range is its slot.  Key j of (slot, quarter) of row i sits
// at ((slot * 4 + quarter) * K + j) * ldl + i: consecutive rows are adjacent, so a
// warp's writes and the merge kernel's reads are coalesced.
__host__ __device__ inline int64_t topk_list_index(int32_t slot, int32_t quarter, int32_t j, int32_t K, int32_t ldl,
                                                   int32_t row) {
  return (static_cast<int64_t>(slot * 4 + quarter) * K + j) * ldl + row;
}

struct TopkMergeParams {
  const unsigned long long* lists;
  int32_t n_a, n_b, ldl, npieces, k;  // npieces: of the row problem; k <= K: entries written per row
  int32_t* scores;                 // [n_a][k]
  int32_t* index;                  // [n_a][k]
  int32_t* status;                 // SERAC_OK, or SERAC_ETIMEOUT when a kernel wait ran out (may be NULL)
  const int32_t* err;
};

// Final top-2 of a row or column as two 64-bit keys (best, second):
// key = score << 32 | (0xFFFFFFFF - index), 0 = empty.  A plain unsigned max orders
// by score, then lower index.  Kernels merge into them with atomicMax.
constexpr int MAX_PROBLEMS = 2 * MAX_PAIRS;
struct FusedParams {
  int32_t n_pairs;                   // row problems in the launch
  int32_t grid;
  int32_t dump_ld;                   // score-dump row stride (dump mode only)
  int32_t* err;                      // error bits
  int32_t* dump;                     // score dump (dump mode only)
  uint32_t key_mult;                 // 256, read as a kernel parameter (see the epilogue)
  int32_t no_copies;                 // test hook: the producer issues no copies (bounded waits run out)
  int32_t early_dependents;          // let the match launch start beside this kernel's CTAs
  FusedPair pairs[MAX_PROBLEMS];
};

struct StageImage {
  const uint8_t* src;
  int32_t n;
  int32_t row0;  // first staged row
};

struct StageParams {
  int32_t n_images;
  int32_t zero_blocks;   // blocks of the extra grid row that clears `zero`
  uint16_t* staged;      // bf16 bits, [rows][128]
  uint4* zero;           // cleared before the fused kernel (key arrays)
  int64_t zero_n;        // 16-byte words to clear
  int32_t* err;          // error word, cleared too
  StageImage images[512];
};

struct FinishPair {
  int32_t n_a, n_b;
  int32_t row_base;   // first entry of this pair in rowkeys
  int32_t col_base;   // first entry of this pair in colkeys
  int32_t blk_base;   // first block (and status word) of this pair in the match launch
  int32_t nblk;       // blocks of this pair (MATCH_ROWS_PER_BLOCK rows each, at least 1)
  int32_t* matches;
  int32_t* count;
  int32_t* row_top2;
  int32_t* col_top2;
  int32_t capacity;
  int32_t pad_;
};

constexpr int MATCH_THREADS = 128;
constexpr int MATCH_ROWS_PER_THREAD = 2;
constexpr int MATCH_ROWS_PER_BLOCK = MATCH_THREADS * MATCH_ROWS_PER_THREAD;

struct FinishParams {
  int32_t n_pairs;
  int32_t total_blocks;
  int32_t ratio_num_sq, ratio_den_sq, norm_sq, min_score, mutual, col_ratio;
  const unsigned long long* rowkeys;
  const unsigned long long* colkeys;
  int32_t* tickets;               // [pair]: next block index of the pair (zeroed)
  unsigned long long* status;     // [block]: look-back word (zeroed)
  uint4* zero;                    // the other chunk's key region, cleared here
  int64_t zero_n;                 // 16-byte words
  int32_t* err;
  FinishPair pairs[MAX_PAIRS];
};

// launchers (defined in fused.cu / finish.cu); return a cudaError_t value
int launch_stage(const StageParams& p, int64_t max_chunks, void* stream, bool beside_fused);
int launch_fused(const FusedParams& p, const void* tmap, int mode, void* stream);
int launch_topk_merge(const TopkMergeParams& p, int K, void* stream);
int launch_match(const FinishParams& p, void* stream);
int fused_smem_bytes();

}  // namespace serac
