/*
 * sgemm_gb300.h -- C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * The operation is the one every kernel on the pages computes:
 *   C = alpha * A * B + beta * C
 * on row-major FP32 matrices ("Shared Memory Tiling", kernel listing, final
 * store alpha * acc + beta * C; "Warp Tiling: A Third Level of Tiling",
 * section "The Kernel", epilogue; "Vectorized Memory Access: 128-bit Loads and
 * Stores", section "The Kernel", epilogue). The pages' kernels take
 * (M, N, K, alpha, A, B, beta, C) with implicit leading dimensions lda = K,
 * ldb = ldc = N; this interface adds explicit leading dimensions and a stream.
 *
 * Layout (row-major): A(i,k) = A[i*lda + k] for i < M, k < K;
 *                     B(k,j) = B[k*ldb + j] for k < K, j < N;
 *                     C(i,j) = C[i*ldc + j] for i < M, j < N.
 * Elements outside those ranges (padding between rows) are never read or
 * written.
 *
 * Ownership: all matrix pointers are DEVICE pointers owned by the caller. The
 * library owns only a small per-(device, stream) workspace (split-K partial
 * tiles, their flags and a device status word), allocated on first use and
 * released by sgemm_shutdown(). No call here takes a torch type.
 *
 * Errors: every function returns an sgemm_status. Argument errors are found on
 * the host before anything is launched, and leave C untouched. Launch errors
 * are returned synchronously. A kernel that gives up on a bounded wait (a
 * copy, slot or partial that never arrived within the wait limit) records a
 * device status that sgemm_poll_device_status() reports.
 *
 * Threading: calls are asynchronous with respect to the host and ordered on
 * `stream`; the workspace is per (device, stream), so concurrent calls on
 * different streams do not share it. Host-side state is guarded by a mutex.
 *
 * CUDA graphs: sgemm, sgemm_ex, sgemm_strided_batched and sgemm_3xtf32 can be
 * captured into a graph and replayed, once a call of at least the same size
 * has run on the capturing stream outside the capture (it sets the device up
 * and sizes the stream's workspace; a call that would have to grow it during
 * capture returns SGEMM_ERR_CAPTURE and launches nothing). The graph keeps
 * the stream's workspace: do not replay it concurrently with other work on
 * that stream's workspace. sgemm_noalloc needs no workspace at all.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SGEMM_OK = 0,
  SGEMM_ERR_INVALID_DIM = -1,       /* M, N or K negative                        */
  SGEMM_ERR_INVALID_LD = -2,        /* lda < max(1,K), ldb < max(1,N), ldc < max(1,N) */
  SGEMM_ERR_NULL_PTR = -3,          /* a matrix that must be accessed is NULL     */
  SGEMM_ERR_UNSUPPORTED_DEVICE = -4,/* current device is not sm_103               */
  SGEMM_ERR_LAUNCH = -5,            /* CUDA runtime error while launching         */
  SGEMM_ERR_DEVICE_TIMEOUT = -6,    /* a kernel gave up on a bounded wait         */
  SGEMM_ERR_ALLOC = -7,             /* workspace allocation failed                */
  SGEMM_ERR_MISALIGNED = -8,        /* a matrix pointer is not 4-byte aligned     */
  SGEMM_ERR_INVALID_VALUE = -9,     /* other invalid argument (config id, buffer) */
  SGEMM_ERR_NOALLOC_CAPACITY = -10, /* sgemm_noalloc: problem needs more scratch
                                       than its fixed buffer holds             */
  SGEMM_ERR_CAPTURE = -11           /* the per-stream workspace would have to grow
                                       while `stream` is captured into a CUDA
                                       graph (nothing launched; call once on
                                       the stream before capturing)            */
} sgemm_status;

/* Operand forms of sgemm_ex / sgemm_strided_batched (row-major storage). */
typedef enum {
  SGEMM_OP_N = 0, /* the operand as stored                               */
  SGEMM_OP_T = 1  /* its transpose: A stored K x M, or B stored N x K     */
} sgemm_op;

/*
 * C = alpha * A * B + beta * C (FP32, FFMA path).
 *
 * M, N, K >= 0. lda >= max(1, K), ldb >= max(1, N), ldc >= max(1, N).
 * Quick returns: M == 0 or N == 0 does nothing. K == 0 or alpha == 0 scales
 * C by beta without reading A or B. beta == 0 never reads C, so C may hold
 * NaN or garbage. A and B may have any 4-byte alignment (the 128-bit and TMA
 * paths are used only when alignment allows). C must not overlap A or B.
 * stream: a cudaStream_t (NULL = legacy default stream). Problems with
 * M * N * K <= 2^25 run a latency-first kernel (one CTA per 32 x 32 tile, no
 * K-split) unless a tile configuration is forced; larger ones the persistent
 * kernel with the tuned configuration of their shape class.
 * Pages: the result is the one every kernel of "Shared Memory Tiling" (kernel
 * listing, final store), "Vectorized Memory Access: 128-bit Loads and Stores"
 * and "Warp Tiling: A Third Level of Tiling" (section "The Kernel",
 * epilogues) computes. The pages are silent on leading dimensions, shapes that
 * are not tile multiples, alignment, and the beta == 0 / alpha == 0 / K == 0
 * cases; the rules above are the plain BLAS reading of those points.
 */
int sgemm(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
          float beta, float* C, int ldc, void* stream);

/*
 * Opt-in tensor-core path: the same C = alpha * A * B + beta * C, with the
 * same arguments, checks and workspace, computed as three TF32 products per
 * FP32 product on the tcgen05 tensor cores (each operand split into a TF32
 * high part and a TF32 residual; the dropped residual product is below
 * 3 * 2^-20 of sum |a||b|, inside the library's FP32 tolerance, and integer
 * inputs up to 2^11 stay exact). The pages have no tensor-core kernel; this is
 * the split-operand method of Ootomo and Yokota (2022). It uses 4 * N * K
 * bytes of workspace for a transposed copy of B, plus 4 * M * K when the rows
 * of A are not 16-byte aligned (A is then copied). Reported separately from the
 * FFMA path.
 */
int sgemm_3xtf32(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                 int ldb, float beta, float* C, int ldc, void* stream);

/*
 * Kernel form of sgemm_3xtf32 for later calls (process-wide):
 *   SGEMM_X3_PAIR (the default): clusters of two CTAs on vertically adjacent
 *     128 x 256 tiles; the even CTA issues M = 256 MMAs over both
 *     (tcgen05 cta_group::2), each CTA holding its A tile and half of the B
 *     tile in shared memory and its 128 rows of the accumulator in TMEM;
 *   SGEMM_X3_SINGLE: single CTAs, each loading its own A and B tiles.
 * In both forms every CTA loads only its own tiles (no TMA load is shared
 * between CTAs). The pair form runs where the device can co-schedule CTA
 * pairs and the problem has at least two waves of whole tile pairs, else
 * single CTAs. Both give the same results within the tolerance (bit-identical
 * on integer inputs). Returns the previous setting, or
 * SGEMM_ERR_INVALID_VALUE (nothing changed) for another value. The pages are
 * silent (no tensor-core kernel).
 */
#define SGEMM_X3_SINGLE 1
#define SGEMM_X3_PAIR 2
int sgemm_3xtf32_set_kernel_form(int form);

/*
 * The plan sgemm_3xtf32 follows for an M x N x K problem (host arithmetic
 * only, no device needed): `form` is the requested kernel form, `pairs` how
 * many CTA pairs the device keeps resident (0: none), `sms` its SM count.
 * out (9 ints) = {form that runs, k-slice width, stages, CTAs, schedule
 * units (a CTA pair each in the pair forms), whole-tile units, K-split units,
 * k-slices, tile width in N}. The pair form falls back to single CTAs when
 * pairs == 0 or when every tile would be split along K. The tile width: 64
 * for N <= 64 and for problems of few 128-wide tiles ((sms / tiles)^2 >
 * ceil(K / 32) / 2), 128 for N <= 128 and for fewer than two waves of
 * 256-wide tiles with at most 48 slices of 32 of their work per SM, else 256;
 * the 64- and 128-wide tiles run on single CTAs with 32-wide slices.
 * Returns SGEMM_OK, SGEMM_ERR_INVALID_DIM unless
 * M, N, K >= 1 (only such problems launch the GEMM kernel), or
 * SGEMM_ERR_INVALID_VALUE for another form, pairs < 0, sms < 1 or a NULL out.
 * The pages are silent (no tensor-core kernel, one CTA per tile).
 */
int sgemm_3xtf32_plan(int M, int N, int K, int form, int pairs, int sms, int* out);

/*
 * C = alpha * op(A) * op(B) + beta * C, row-major, FFMA path. op(A) is M x K:
 * A itself (SGEMM_OP_N, stored M x K, lda >= max(1, K)) or the transpose of an
 * A stored K x M (SGEMM_OP_T, lda >= max(1, M)); op(B) is K x N: B (stored
 * K x N, ldb >= max(1, N)) or the transpose of a B stored N x K (ldb >=
 * max(1, K)). A stored transposed A arrives by TMA (no transposing copy); a
 * stored transposed B goes through the transposing copy the kernel uses for
 * row-major A. Column-major callers: a column-major M x N result is the
 * row-major N x M result of op(B)^T op(A)^T, i.e. call with the operands and
 * M, N swapped. Otherwise as sgemm(); SGEMM_ERR_INVALID_VALUE for another op.
 * The pages compute row-major A * B only; transposed operands are the BLAS
 * generalisation they never reach (silent).
 */
int sgemm_ex(int opA, int opB, int M, int N, int K, float alpha, const float* A, int lda,
             const float* B, int ldb, float beta, float* C, int ldc, void* stream);

/*
 * `batch` independent products C_i = alpha * op(A_i) * op(B_i) + beta * C_i
 * with A_i = A + i * strideA, B_i = B + i * strideB, C_i = C + i * strideC
 * (strides in elements, >= 0; a zero stride reuses one matrix for every i,
 * which is only valid for A and B). One launch covers every product: the
 * batch index is the outermost tile coordinate of the persistent schedule.
 * C_i must not overlap each other or any A_j, B_j. batch == 0 does nothing.
 * The pages are silent (one product per launch).
 */
int sgemm_strided_batched(int opA, int opB, int M, int N, int K, float alpha, const float* A,
                          int lda, long long strideA, const float* B, int ldb, long long strideB,
                          float beta, float* C, int ldc, long long strideC, int batch,
                          void* stream);

/*
 * The same C = alpha * A * B + beta * C with A, B and C in HOST memory (pinned
 * memory gives full copy bandwidth; pageable memory works but the copies may
 * block the calling thread). K is cut into chunks whose host -> device copies
 * overlap the multiplication of the previous chunk on the GPU (by default the
 * chunks grow geometrically, each as much wider as multiplying a column of K
 * takes longer than copying it); the incoming C (read only when beta != 0)
 * arrives in row panels and is added panel by panel at the end, and each
 * finished row panel is copied back while the next one is computed. All work is queued behind earlier work on
 * `stream`, and `stream` waits for the final copy: once the caller has
 * synchronised `stream`, C holds the result. The host buffers must stay
 * valid until then. Device buffers, two copy streams and their events are
 * owned by the library per (device, stream) and reused by later calls (freed
 * by sgemm_shutdown). Same argument checks and status codes as sgemm().
 * The pages are silent: they time device-resident operands only.
 */
int sgemm_host(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
               float beta, float* C, int ldc, void* stream);

/*
 * Copy/compute pipeline of later sgemm_host calls (process-wide). With
 * mid == 0 (the default) K is cut into geometrically growing chunks: a first
 * chunk of `first` columns (0: 128), each next one min(4, max(1.5,
 * M N / (M + N) / 755)) times wider, a remainder narrower than half the next
 * width joining the chunk before it, and, when last > 0, a last chunk of
 * `last` columns. With mid > 0: a first chunk of `first` columns (0: none;
 * taken only when K >= 2 * first + last), middle chunks of about `mid`
 * columns, and a last chunk of `last` columns (0: as wide as the middle
 * chunks). The last chunk is computed and copied back in `panels` row panels
 * (0: 4; at most 8; fewer when M < 512 * panels). Widths are rounded up to
 * multiples of 32; at most 9 chunks.
 * The result does not depend on the setting beyond the order of the sum
 * over k. Returns SGEMM_ERR_INVALID_VALUE (nothing changed) for a negative
 * value or more than 8 panels. The pages are silent.
 */
int sgemm_host_set_pipeline(int first, int mid, int last, int panels);

/* Human-readable text for a status code (static storage, never NULL). The
 * pages are silent: their kernels return no status. */
const char* sgemm_status_string(int status);

/*
 * Name of the tile configuration and schedule the calling thread's last
 * sgemm() used, copied into buf (at most len bytes, NUL-terminated).
 * Returns SGEMM_OK, or SGEMM_ERR_INVALID_VALUE if buf is NULL or len < 1.
 * The pages name the configuration beside every measurement ("Autotuning:
 * Searching the Tile-Shape Space", section "What The Sweep Found"); this is
 * that name for the library's own choice.
 */
int sgemm_last_config(char* buf, int len);

/*
 * Waits for `stream`, then reports and clears the device status word of this
 * (device, stream) workspace: SGEMM_OK, or SGEMM_ERR_DEVICE_TIMEOUT if a
 * kernel gave up on a bounded wait since the last poll. *detail (if not NULL)
 * receives the device-side code (1 = operand tile, 2 = slot release, 3 =
 * split partial, 4 = CTA rendezvous, 5 = the two CTAs of a two-SM pair of
 * sgemm_3xtf32 got different tensor-memory columns; none of them is a device
 * fault, and the context stays usable). SGEMM_ERR_LAUNCH if synchronising
 * fails. `detail` extends the one-argument form this call would otherwise have: the
 * status alone cannot say which wait gave up. The pages are silent (their
 * kernels have no bounded waits and report nothing).
 */
int sgemm_poll_device_status(void* stream, int* detail);

/* Frees every workspace, device buffer, stream and event the library
 * allocated (after synchronising the device). Later calls allocate again.
 * The pages are silent (their kernels allocate nothing). */
void sgemm_shutdown(void);

/*
 * Tile configurations compiled into the library. sgemm_config_count() gives
 * their number; sgemm_config_info() fills name (len bytes) and the tile
 * parameters of configuration `id` as
 * {BM, BN, BK, WM, WN, WNITER, TM, TN, NT, STAGES, MINB, KU, ORDER} in
 * params[13] (KU: k-steps per unrolled chunk; ORDER: 0 row-by-row FFMA, 1 zig-zag
 * FFMA, 2 paired FMA, 3 paired FMA column by column).
 * Pages: the tuple of "Autotuning: Searching the Tile-Shape Space", section
 * "Mechanics" (the kernel's template parameters), plus this kernel's own
 * pipeline depth, residency, unroll and FMA order.
 */
int sgemm_config_count(void);
int sgemm_config_info(int id, char* name, int len, int* params);

/*
 * Forces every later sgemm() on this process to use configuration `id`
 * (-1 restores the automatic per-shape choice). For tuning and tests; the
 * sweep of "Autotuning: Searching the Tile-Shape Space" ("Mechanics") times
 * one configuration at a time in the same way.
 */
int sgemm_force_config(int id);

/*
 * How row-major A reaches shared memory in later calls (process-wide).
 * The staged variant: where the configuration is built with it (32-wide
 * k-slices, at most 64 accumulators per lane), B arrives by TMA and A is
 * 16-byte aligned with lda (and, batched, the matrix stride) a multiple of 4,
 * one TMA box per k-slice copies A as it is stored into a staging slot and
 * one extra producer warp transposes it into the padded As[k][m], so the FMA
 * warps issue no copies. Otherwise every thread issues the transposing
 * 4-byte copy ("Vectorized Memory Access: 128-bit Loads and Stores", section
 * "Why As Has To Be Transposed"; the pages copy with the FMA threads).
 * on = 1 (the default): the staged variant where allowed and each CTA runs
 * at least 8 k-slices on average (below that its extra step of latency
 * costs more than it saves); 2: wherever allowed, whatever the size; 0:
 * never. Both fill the same As[k][m] and sum in the same order, so results
 * are bit-identical. Returns the previous setting, or
 * SGEMM_ERR_INVALID_VALUE (nothing changed) for another value.
 */
int sgemm_set_staged_a(int on);

/*
 * 1 when tile configuration `id` is built for every operand layout (op(A),
 * op(B) in {N, T}; sgemm_ex and sgemm_strided_batched can use it), 0 when
 * only for row-major A and B, SGEMM_ERR_INVALID_VALUE for an unknown id.
 * The pages are silent (row-major operands only).
 */
int sgemm_config_layouts(int id);

/*
 * The configuration sgemm() picks by itself for an M x N x K problem (the
 * tuned table's entry for the problem's shape class, ignoring
 * sgemm_force_config). *shape_class (if not NULL) receives the class:
 * 0 square-large (M * N >= 12 Mi), 1 square-small (M * N < 3 Mi),
 * 2 K-dominant (K >= 4 max(M, N)), 3 N <= 96, 4 M <= 96, 5 tiny (at most
 * 2^28 multiply-adds), 6 square-mid (3 Mi <= M * N < 12 Mi).
 * Returns the configuration id or SGEMM_ERR_INVALID_DIM. Host only.
 * Pages: "Autotuning: Searching the Tile-Shape Space" picks one configuration
 * by measurement for one shape ("What The Sweep Found") and notes that the
 * winner depends on the shape ("What Could Be Improved"); this repeats the
 * search per shape class.
 */
int sgemm_choose_config(int M, int N, int K, int* shape_class);

/*
 * The legality checker of the tile configurations, evaluated on the host:
 * 0 if the tuple is legal for the FFMA kernel, else the number of the first
 * rule it breaks. params = {BM, BN, BK, WM, WN, WNITER, TM, TN, NT, STAGES,
 * MINB, KU, ORDER}. derived (if not NULL) receives {WMITER, WSUBM, WSUBN, accumulators
 * per thread, shared bytes per CTA} when the tuple is legal.
 * Pages: "Autotuning: Searching the Tile-Shape Space", sections "Most
 * Configurations Are Not Wrong By A Little" (the kernel's unstated
 * assumptions) and "Mechanics" (a compile-time legality gate); the rules here
 * are this kernel's own assumptions.
 */
int sgemm_cfg_check(const int* params, int* derived);

/*
 * The persistent schedule sgemm() would use for an M x N x K problem with
 * configuration `id` on `capacity` resident CTAs (host arithmetic only, no
 * device needed), under the policy sgemm() would take (a forced one, else
 * the tuned policy of the problem's shape class). out = {tiles_m, tiles_n,
 * kiters, grid, dp_tiles, sk_q, sk_r, group_m}. Returns SGEMM_OK or an
 * argument error.
 * The pages launch one CTA per C tile ("Shared Memory Tiling", kernel launch
 * grid); the persistent schedule is this library's (silent on the pages).
 */
int sgemm_schedule_query(int M, int N, int K, int id, int capacity, int* out);

/*
 * Persistent-schedule policies (the values of policy[0]):
 *   SGEMM_SCHED_HYBRID      whole tiles, then the last one to two waves' worth
 *                           of tiles split into k-slice units (with fewer
 *                           tiles than CTA slots, every tile is split);
 *   SGEMM_SCHED_HYBRID_TAIL whole waves of whole tiles; only the ragged last
 *                           wave is split;
 *   SGEMM_SCHED_DATA_PARALLEL whole tiles only;
 *   SGEMM_SCHED_STREAM_K    every tile split, the k-slice units spread evenly;
 *   SGEMM_SCHED_SPLIT_K     every tile cut into policy[3] equal k-ranges.
 * A policy is int[4] = {mode, raster group height in tiles (>= 1), fewest
 * k-slices per CTA when splitting (>= 1), splits (>= 1)}. Every policy gives
 * a correct result; split partial sums are added in a fixed order, so a
 * policy always gives the same bits. The pages are silent (one CTA per tile).
 */
#define SGEMM_SCHED_HYBRID 0
#define SGEMM_SCHED_HYBRID_TAIL 1
#define SGEMM_SCHED_DATA_PARALLEL 2
#define SGEMM_SCHED_STREAM_K 3
#define SGEMM_SCHED_SPLIT_K 4

/*
 * The schedule of an M x N x K problem with BM x BN tiles and BK-wide
 * k-slices on `capacity` CTA slots under `policy` (host arithmetic only):
 * out as for sgemm_schedule_query. Returns SGEMM_OK, SGEMM_ERR_INVALID_DIM
 * (negative size, or more than 2^31 - 1 tiles) or SGEMM_ERR_INVALID_VALUE.
 */
int sgemm_schedule_plan(int M, int N, int K, int BM, int BN, int BK, int capacity,
                        const int* policy, int* out);

/*
 * Forces `policy` on every later sgemm(), sgemm_ex() and
 * sgemm_strided_batched() call of this process (the tuner and tests); NULL or
 * policy[0] < 0 restores the tuned policy of each problem's shape class.
 * Returns SGEMM_OK or SGEMM_ERR_INVALID_VALUE (nothing changed).
 */
int sgemm_force_schedule(const int* policy);

/*
 * The tuned policy sgemm() uses by itself for an M x N x K problem (that of
 * its shape class), written to policy[4]. Returns SGEMM_OK or an argument
 * error. Host only.
 */
int sgemm_choose_policy(int M, int N, int K, int* policy);

/*
 * Piece `i` of CTA `b` under the schedule {tiles_m, tiles_n, kiters, grid,
 * dp_tiles, sk_q, sk_r, group_m} (as returned above): out = {tile, kb, ke,
 * tile_m, tile_n, contributors, is_partial}. Returns the number of pieces of
 * CTA b, or a negative status. Host arithmetic only. Pages: silent (see
 * sgemm_schedule_query).
 */
int sgemm_schedule_piece(const int* sched, int b, int i, int* out);

/*
 * Diagnostic: launches one CTA that waits on a shared-memory barrier nothing
 * ever arrives on, with a limit of timeout_ns, through the same bounded wait
 * the GEMM kernels use. The wait must run out and record device code 1; read
 * it with sgemm_poll_device_status(). Nothing faults and nothing hangs.
 * The pages are silent.
 */
int sgemm_diag_wait_timeout(long long timeout_ns, void* stream);

/* Upper bound, in nanoseconds, of every wait inside the kernels (default
 * 4e9). Values < 1000 are rejected. Returns the previous value or a negative
 * status. The pages are silent. */
long long sgemm_set_wait_timeout_ns(long long ns);

/*
 * Diagnostic: the TF32 tensor-core throughput of the current device, in
 * TFLOP/s, measured. One CTA per SM issues `iters` x 4 back-to-back
 * tcgen05.mma.kind::tf32 of M 128, N 256, K 8 from shared memory into tensor
 * memory, with no loads in the loop; the launch is timed with CUDA events
 * (about 6 ms at iters = 20000 on GB300). Synchronous. The 3xTF32 path's
 * roofline divides this by three. Returns SGEMM_ERR_INVALID_VALUE for iters
 * < 1 or a NULL result pointer, SGEMM_ERR_DEVICE_TIMEOUT if the MMAs did not
 * complete within 4 s. The pages are silent (no tensor-core kernel).
 */
int sgemm_diag_tf32_mma_rate(int iters, double* tflops);

/*
 * Diagnostic: the same measurement for the pair form the 3xTF32 path runs by
 * default. Clusters of two CTAs (as many as are resident at once); the even
 * CTA issues `iters` x 4 tcgen05.mma.cta_group::2.kind::tf32 of M 256 (128
 * rows per CTA), N 256 (half of B in each CTA), K 8. The rate counts the
 * multiply-adds of all SMs taking part. Same arguments, errors and duration
 * as sgemm_diag_tf32_mma_rate. The pages are silent.
 */
int sgemm_diag_tf32_pair_mma_rate(int iters, double* tflops);

/*
 * The same C = alpha * A * B + beta * C as sgemm(), with the same arguments,
 * checks and results, for callers that must not allocate device memory: code
 * running while a stream is captured into a graph, applications whose memory
 * pool owns every free byte and forbids hidden allocations, and latency-bound
 * loops that cannot absorb an allocation. The pages have no counterpart; this
 * is a packaging of the same kernel.
 *
 * The kernel's scratch (status word, one flag per persistent CTA, split-K
 * partial tiles) lives in one fixed 24 MiB device array inside the library,
 * which every GPU that loads the library holds until the process exits; no
 * call allocates. The first call on a device does the set-up (the array's
 * device address, the kernels' attributes): make it before any stream
 * capture. A problem whose schedule needs more scratch than the array holds
 * returns SGEMM_ERR_NOALLOC_CAPACITY and launches nothing (on a 152-SM GB300
 * every problem fits). All calls share the array: calls that overlap on the
 * GPU (other streams, other host threads) race and must not be issued. Every
 * wait inside the kernel is bounded by the library's wait limit
 * (sgemm_set_wait_timeout_ns). A kernel that gives up records its code in the
 * array, where it stays until sgemm_noalloc_poll_status() reads it
 * (sgemm_poll_device_status() reports only the per-stream workspaces). The
 * tile configuration is always the automatic choice (sgemm_force_config()
 * does not apply), and problems with M * N * K <= 2^25 run the same
 * tiny-problem kernel as sgemm().
 */
int sgemm_noalloc(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                  int ldb, float beta, float* C, int ldc, void* stream);

/*
 * Waits for `stream`, then reports and clears the device status that
 * sgemm_noalloc calls on the current device recorded in the library's fixed
 * array: SGEMM_OK, or SGEMM_ERR_DEVICE_TIMEOUT with *detail (if not NULL)
 * set to the code (the same codes as sgemm_poll_device_status). After a
 * timeout it also clears the array's split-K flags, which an aborted call can
 * leave published. Allocates nothing. SGEMM_OK when sgemm_noalloc has not
 * run on this device; SGEMM_ERR_LAUNCH if synchronising or a copy fails.
 * The pages have no counterpart (they report no device-side errors).
 */
int sgemm_noalloc_poll_status(void* stream, int* detail);

/*
 * Three kernels of the pages' series, rebuilt for this GPU to measure what
 * each technique buys; sgemm() never uses them:
 *   kernel 3 -- shared-memory tiling ("Shared Memory Tiling"): 32 x 32 C tile
 *               per CTA of 1024 threads, one output per thread;
 *   kernel 7 -- vectorized 2-D block tiling ("Vectorized Memory Access:
 *               128-bit Loads and Stores"): 128 x 128 C tile, BK = 8, 8 x 8
 *               outputs per thread, 128-bit loads, A transposed in shared
 *               memory;
 *   kernel 8 -- warp tiling ("Warp Tiling: A Third Level of Tiling"):
 *               128 x 64 C tile, BK = 16, 64 x 32 warp tiles of 2 x 2
 *               sub-tiles, 4 x 4 outputs per thread and sub-tile.
 * Arguments after `kernel`, their checks, the quick returns and the result
 * are those of sgemm(): any shape, leading dimension and 4-byte alignment
 * (128-bit accesses are used only when A, B and C are 16-byte aligned and
 * lda, ldb, ldc are multiples of 4). One CTA per C tile on `stream`; no
 * workspace and no device status. kernel other than 3, 7 or 8 returns
 * SGEMM_ERR_INVALID_VALUE; more than 2^31 - 1 tiles SGEMM_ERR_INVALID_DIM.
 */
int sgemm_ladder(int kernel, int M, int N, int K, float alpha, const float* A, int lda,
                 const float* B, int ldb, float beta, float* C, int ldc, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
