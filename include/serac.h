/*
 * serac.h -- C ABI of libserac_gb300.so: exhaustive SIFT descriptor matching with a
 * fused top-2 on GB300 (sm_103a).
 *
 * What is computed (the method of the "SERAC" page -- a fused descriptor matcher for
 * COLMAP -- sections "What changed" and "Exactness"):
 *
 *   s(i, j) = sum_{k<128} a[i][k] * b[j][k]      exact integer, 0 <= s <= 8,323,200
 *
 *   row top-2    (s1, j1, s2, j2) of row i: the two best positive scores of the row,
 *                ordered by score descending then column ascending, each padded with
 *                (0, -1) ("Exactness": identity (0, -1, 0), zero floor, smallest
 *                column on an exact top-1 tie);
 *   column top-2 (c1, i1, c2, i2) of column j: the same over rows ("GPU kernel time":
 *                the column direction, ColMatch, feeds the cross check);
 *   test(t)      t.j1 >= 0  and  den * (N - t.s1) < num * (N - t.s2)  and
 *                t.s1 >= min_score   (evaluated in 64-bit integers; the page fixes
 *                only max_ratio <= 1, default 0.8, and that a tie rejects -- this is
 *                the chord-distance ratio squared, r^2 = num/den, N = 512^2);
 *   match        (i, j1(i)) is kept iff test(row i) and, when `mutual`, i1(j1(i)) == i,
 *                and, when `col_ratio`, test(column j1(i)).  Matches are listed by
 *                ascending i.
 *
 * The similarity matrix is never stored ("Fused row reduction": only the top two
 * scores of each row and column survive); the contraction runs on the tcgen05
 * tensor cores with f32 accumulation, exact because every partial sum is an
 * integer below 2^24.
 *
 * Conventions for every entry point:
 *   - descriptor arrays are n x 128 uint8, row-major, contiguous, 16-byte aligned,
 *     read only, in memory the GPU can address: device memory, or pinned host memory
 *     (cudaHostAlloc / cudaHostRegister; the staging kernel then reads it over the
 *     host link, so no separate host-to-device copy is needed);
 *   - outputs are caller-owned, in device memory or pinned host memory (the kernels
 *     then write the results straight to the host); the workspace is device memory;
 *   - calls are asynchronous on `cuda_stream` (a cudaStream_t; NULL = legacy default
 *     stream); results are valid once that stream has synchronised;
 *   - a call returns a status below; a negative status means nothing was enqueued;
 *   - sizes: 0 <= n <= SERAC_MAX_N per image.
 *
 * Errors found by the GPU (a bounded wait that ran out inside a kernel) are reported
 * through `*count`, which then holds a negative status instead of a match count.
 */
#ifndef SERAC_H
#define SERAC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SERAC_DIM 128
#define SERAC_MAX_N (1 << 24)

/* status codes */
#define SERAC_OK 0
#define SERAC_EINVAL (-1)        /* bad argument: null pointer, n out of range, misaligned */
#define SERAC_ECAPACITY (-2)     /* (reported through count > capacity; never returned) */
#define SERAC_ECUDA (-3)         /* a CUDA runtime call failed */
#define SERAC_ETIMEOUT (-4)      /* a bounded wait inside a kernel ran out (via *count) */
#define SERAC_EWORKSPACE (-5)    /* workspace missing or smaller than the size query */
#define SERAC_EUNSUPPORTED (-6)  /* current device is not sm_103 or TMA encoding unavailable */

/* Matching parameters, exact integers.  serac_default_params fills them from the
 * page's knobs (max_ratio 0.8, max angle 0.7 rad -> 16/25, N = 262144, 200499; no
 * feature cap). */
typedef struct {
  int32_t ratio_num_sq; /* r^2 = num / den (0.8 -> 16) */
  int32_t ratio_den_sq; /*                 (0.8 -> 25) */
  int32_t norm_sq;      /* N, squared norm of a unit descriptor at scale 512: 262144 */
  int32_t min_score;    /* distance gate: s1 >= ceil(cos(max_angle) * N) */
  int32_t mutual;       /* 1: require i1(j1(i)) == i */
  int32_t col_ratio;    /* 1: column j1(i) must pass the same test */
  int32_t max_features; /* feature cap K ("Memory": the match cap clamps away the
                           features past it): K > 0 matches only the first K
                           descriptors of each image, exactly as if the caller had
                           passed n = min(n, K); 0 = no cap */
} serac_params;

/* One image pair for match_batch (device pointers, as for match_pair). */
typedef struct {
  const uint8_t* a;
  int32_t n_a;
  const uint8_t* b;
  int32_t n_b;
} serac_pair;

/* Outputs of one pair (device pointers, owned by the caller).
 *   matches  [capacity][2] int32 (i, j), ascending i; at most `capacity` are written
 *   count    1 int32: the total number of matches (may exceed capacity: then only the
 *            first `capacity` were written) or a negative status from the GPU;
 *            capacity n_a always suffices (min(n_a, n_b) when `mutual` is set)
 *   row_top2 optional (NULL to skip): [n_a][4] int32 (s1, j1, s2, j2)
 *   col_top2 optional (NULL to skip): [n_b][4] int32 (c1, i1, c2, i2)
 * Under a feature cap K (serac_params.max_features) read n_a and n_b above as
 * min(n_a, K) and min(n_b, K): nothing past them is written. */
typedef struct {
  int32_t* matches;
  int32_t capacity;
  int32_t* count;
  int32_t* row_top2;
  int32_t* col_top2;
} serac_out;

/* Fill `p` from a ratio (read to 4 decimals, squared and reduced to num/den) and a
 * maximum angle in radians (min_score = ceil(cos(angle) * 262144)); mutual = 1,
 * col_ratio = 1, max_features = 0.  Host only.  Returns SERAC_EINVAL if p is NULL, max_ratio is not in
 * (0, 1] or the angle is not in [0, pi/2]. */
int serac_default_params(serac_params* p, float max_ratio, float max_angle_rad);

/* Workspace bytes match_pair needs for these sizes (host only; never fails). */
size_t serac_pair_workspace_size(int32_t n_a, int32_t n_b);

/* Match one pair (the method above).  `workspace` is device memory of at least
 * serac_pair_workspace_size(n_a, n_b) bytes, 256-byte aligned; its contents need no
 * initialisation and are scratch for this call (calls sharing a workspace must not
 * overlap on the GPU).  Returns SERAC_OK once all kernels are enqueued. */
int match_pair(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b,
               const serac_params* params, const serac_out* out,
               void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Workspace bytes match_batch needs for these pairs (host only).  Images that appear
 * in several pairs (same pointer and size) are staged once. */
size_t match_batch_workspace_size(const serac_pair* pairs, int32_t n_pairs);

/* Match every pair of `pairs` (host array) into outs[k] (host array of device
 * outputs).  Equivalent to match_pair on each pair in turn, scheduled as a few
 * persistent launches over all pairs' tiles.  Same workspace rules as match_pair.
 * The pairs run in launch chunks of at most 128; each chunk's images are staged
 * before its launch, the later chunks' on an internal per-thread stream while the
 * earlier chunks compute (the call still only orders work on `cuda_stream`: the
 * internal stream starts after the work already queued there, and the launches that
 * need its staging wait for it). */
int match_batch(const serac_pair* pairs, int32_t n_pairs, const serac_params* params,
                const serac_out* outs, void* workspace, size_t workspace_bytes,
                void* cuda_stream);

/* The full score matrix S[n_a][n_b] (int32, device, row stride n_b) computed by the
 * same tensor-core tiles as match_pair, written out instead of reduced: a check of
 * the contraction's exactness and of "fused == unfused".  For small n only (the
 * output is n_a * n_b * 4 bytes).  Same workspace size as match_pair. */
int serac_scores(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b,
                 int32_t* scores, void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Row top-k for guided matching (k = 1..SERAC_MAX_TOPK): for every row i of A, the k
 * highest-scoring columns of B, in the order of the method's candidate list -- score
 * descending, then lower column first, zero scores excluded ("SERAC" page,
 * "Exactness"; the pages keep k = 2, "Real-Time Dense Stereo at 34 Hz on a Jetson TX2
 * (MASDA, Part 3)" on the two scored candidates per pixel) -- padded with (0, -1).
 * scores[i * k + q] and index[i * k + q] (int32, device or pinned host memory, 4-byte
 * aligned) get entry q of row i; for k = 2 they equal the (s1, s2) and (j1, j2) of
 * match_pair's row top-2.  No ratio test or cross check is applied: the list is the
 * candidate set for a later geometric (guided) test.  `status` (int32, device or
 * pinned host, may be NULL) receives SERAC_OK, or SERAC_ETIMEOUT when a bounded wait
 * inside a kernel ran out (then scores and index are not valid), once the stream has
 * run the call.  Workspace: device memory of at least serac_topk_workspace_size(n_a,
 * n_b, k) bytes, 256-byte aligned, scratch for this call.  Argument errors:
 * SERAC_EINVAL (k outside 1..SERAC_MAX_TOPK, sizes outside 0..SERAC_MAX_N, NULL or
 * misaligned pointers), SERAC_EWORKSPACE, SERAC_ECUDA, SERAC_EUNSUPPORTED. */
#define SERAC_MAX_TOPK 8

/* Workspace bytes serac_topk_pair needs on the current device (the split of the work
 * over the device's SMs sets it); 0 if the device cannot be queried or an argument is
 * out of range.  Host only. */
size_t serac_topk_workspace_size(int32_t n_a, int32_t n_b, int32_t k);

int serac_topk_pair(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b, int32_t k,
                    int32_t* scores, int32_t* index, int32_t* status, void* workspace, size_t workspace_bytes,
                    void* cuda_stream);

/* Profiling hook: when both events are non-NULL (cudaEvent_t), every following
 * match_pair / match_batch / serac_topk_pair call made by the calling thread records `ev_begin` just
 * before its first fused GEMM + top-2 launch and `ev_end` just after it, on the
 * call's stream.  NULL, NULL turns it off.  The setting belongs to the calling
 * thread; other threads' calls are not affected. */
int serac_set_profile_events(void* ev_begin, void* ev_end);

/* SERAC_OK if the current CUDA device is an sm_103 part this library was built for,
 * else SERAC_EUNSUPPORTED (or SERAC_ECUDA if no device can be queried). */
int serac_device_check(void);

/* Number of kernel launches the calling thread's last match_pair / match_batch call
 * enqueued (host-side count, for benchmarking). */
int serac_last_launch_count(void);

/* The cudaError_t value behind the last SERAC_ECUDA this library returned to the
 * calling thread (0 if none), for diagnostics. */
int serac_last_cuda_error(void);

/* Failure-detection test hook.  With enable != 0, the next match_pair / match_batch
 * call (its first fused launch only) runs with a TMA producer that issues no copies:
 * the MMA thread's bounded wait on the operands runs out after its limit (2 s of GPU
 * time), the kernel records the timeout in the error word and winds down, and the
 * call reports SERAC_ETIMEOUT through *count; its other outputs are not valid.  No
 * fault, trap or unbounded wait is involved and the context stays usable: the next
 * call runs normally.  The flag belongs to the calling thread and is consumed by its
 * next call; enable = 0 clears it.  Host only; always returns SERAC_OK. */
int serac_test_inject_timeout(int enable);

/* Size of the library's built-in scratch used by match_pair_noalloc (16 MiB). */
#define SERAC_NOALLOC_SCRATCH_BYTES (16 << 20)

/* match_pair without a workspace argument, for callers that may not allocate
 * device memory: code running inside a host application that owns every device
 * allocation, real-time loops where an allocation's implicit synchronisation or
 * failure is not acceptable, tools that must keep a fixed device footprint.  The
 * paper has no counterpart; it is a deployment convenience.
 *
 * Scratch is one fixed array of SERAC_NOALLOC_SCRATCH_BYTES inside the library
 * (every GPU that loads the library holds it until the process exits).  The call
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   - n_a or n_b outside 0..SERAC_MAX_N (or a NULL / invalid `params`) gives
 *     SERAC_EINVAL; pairs whose serac_pair_workspace_size (of the sizes after the
 *     feature cap) exceeds the scratch are rejected with SERAC_EWORKSPACE (pairs up
 *     to 16,384 x 16,384 fit).
 *   - The first call in each CUDA context looks up the scratch's device address
 *     (cudaGetSymbolAddress) with that context's device current and caches it for
 *     that context (keyed by the context's unique ID); make that first call before
 *     any stream capture.  After cudaDeviceReset, or in another context on the same
 *     device, the module lives at another address: the new context's first call
 *     looks it up again (so, again, make it before any capture in that context).
 *   - All calls share the one scratch array, which keeps the previous call's
 *     contents (the call clears what must start at zero).  Calls that overlap on the
 *     GPU (other streams, other host threads) race on it: serialise them.
 * Arguments, outputs, asynchrony and results are those of match_pair. */
int match_pair_noalloc(const uint8_t* desc_a, int32_t n_a, const uint8_t* desc_b, int32_t n_b,
                       const serac_params* params, const serac_out* out, void* cuda_stream);

/* Host-only view of the work schedule (no GPU needed).  Every pair is matched as two
 * row problems -- the rows of A against the columns B, and the rows of B against the
 * columns A (the pair's column top-2) -- each cut into 128 x 256 tiles.  For `pairs`
 * (pointers are used only to recognise shared images) and at most `grid` persistent
 * CTAs (1..256), report the number of launch chunks and, for the first chunk, the
 * total number of pieces, the pieces of each problem (out_npieces[2 x pairs of that
 * chunk]: entry 2k for pair k's A rows, 2k + 1 for its B rows; a problem's tiles are
 * cut into that many runs of consecutive tiles, each run on its own CTA, 0 for an
 * empty problem -- one run per CTA for a single large pair, whole row tiles for a chunk
 * of many equal pairs, whichever a cost model of the CTAs' loads and segment starts
 * prefers) and the tiles each CTA processes (cta_tiles[grid]; CTAs beyond the chunk's
 * launch grid, which has at most one CTA per tile, get 0).  Any output may be NULL.
 * Returns SERAC_EINVAL on bad input. */
int serac_schedule_describe(const serac_pair* pairs, int32_t n_pairs, int32_t grid, int32_t* out_chunks,
                            int32_t* out_pieces, int32_t* out_npieces, int32_t* cta_tiles);

/* Static text for a status code. */
const char* serac_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* SERAC_H */
