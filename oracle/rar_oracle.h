/*
 * rar_oracle.h -- plain, slow CPU oracle for the ring all-reduce.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include,
 * link or call this code: it exists so that tests, the smoke check and the
 * benchmark's CPU-baseline leg can check the CUDA engines against an
 * independent restatement of the method.  It shares no code, header, table
 * or helper with the CUDA library.
 *
 * Sources restated here (page title, then section):
 *   - "Ring All-Reduce, in depth", section "The schedule": ranks in a logical
 *     ring; reduce-scatter step s, rank r sends chunk (r - s) mod p to r + 1,
 *     which adds it into its own copy; afterwards rank r holds the full sum of
 *     chunk (r + 1) mod p; all-gather step s, rank r sends chunk
 *     (r + 1 - s) mod p and the receiver overwrites.
 *   - same page, section "An implementation": chunk_bounds (the first
 *     N mod p chunks get one extra element) and the simulator in which every
 *     step's sends are snapshotted first and then applied ("all at once").
 *   - same page, section "What real libraries add", paragraph
 *     "Bidirectional rings": a second ring in the opposite direction on half
 *     of the data.
 *   - "AllReduce 与 Ring 通信算法详解", section "AllReduce 语义": the reduction
 *     may be a sum, an average or a maximum.
 *   - "Derive the cost of a ring all-reduce", last probe ("Does the reduction
 *     arithmetic ever matter?"): the reduction runs in the buffer's dtype,
 *     so every hop rounds to that dtype.
 *
 * Element types and ops (codes are the oracle's own):
 *   dtype: ORC_I32 = 0, ORC_F32 = 1, ORC_BF16 = 2, ORC_F16 = 3
 *   op:    ORC_SUM = 0, ORC_MAX = 1, ORC_AVG = 2 (float types only),
 *          ORC_AVG_PREDIV = 3 (float types only): every rank's contribution
 *          is multiplied by 1/p, rounded to the dtype, before the ring-order
 *          sum ("Ring All-Reduce, in depth", "Failure modes": pre-divide so
 *          that a sum over many ranks cannot overflow)
 * Buffers are arrays of the element type in host memory; bf16 and f16 are
 * passed as their raw 16-bit patterns.
 */
#ifndef RAR_ORACLE_H
#define RAR_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_I32 = 0, ORC_F32 = 1, ORC_BF16 = 2, ORC_F16 = 3 };
enum { ORC_SUM = 0, ORC_MAX = 1, ORC_AVG = 2, ORC_AVG_PREDIV = 3 };

/* Ring direction for the simulator and the per-element fold. */
enum { ORC_FORWARD = 0,   /* rank r sends to r + 1 (the pages' ring)            */
       ORC_MIRRORED = 1   /* rank r sends to r - 1 (the opposite-direction ring) */ };

/* chunk_bounds(n, p): starts[0..p], chunk c = [starts[c], starts[c+1]). */
void orc_chunk_bounds(int64_t n, int p, int64_t *starts);

/* Element size in bytes of a dtype code, 0 if unknown. */
int orc_elem_size(int dtype);

/* Round-to-nearest-even conversions, written from the IEEE 754 definition. */
uint16_t orc_f32_to_bf16(float f);
float    orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float f);
float    orc_f16_to_f32(uint16_t h);

/* One hop of the reduction: the running value `acc` arriving from the left
 * neighbour meets the receiver's own element `own`.  Writes op(acc, own)
 * rounded to the dtype into *out.  All three point at one element. */
void orc_combine(int dtype, int op, const void *acc, const void *own, void *out);

/* The schedule simulator.
 *   bufs      p host pointers, each to n elements, modified in place
 *   direction ORC_FORWARD or ORC_MIRRORED
 *   first_step, n_steps
 *             which schedule steps to run: steps 0 .. p-2 are reduce-scatter,
 *             p-1 .. 2p-3 are all-gather; (0, 2p-2) is the whole all-reduce,
 *             (0, p-1) the reduce-scatter alone, (p-1, p-1) the all-gather
 *             alone.  For op ORC_AVG the owner scales its chunk by 1/p right
 *             after the last reduce-scatter step (step p-2), if that step ran;
 *             for ORC_AVG_PREDIV every rank scales its own buffer by 1/p
 *             before step 0, if step 0 runs.
 *   sends     nullable; p counters, incremented by the elements each rank sent
 * Returns 0, or -1 on bad arguments.  p == 1 and n == 0 are no-ops. */
int orc_ring_simulate(void *const *bufs, int p, int64_t n, int dtype, int op,
                      int direction, int first_step, int n_steps,
                      int64_t *sends);

/* The bidirectional variant: [0, n) is split by chunk_bounds(n, 2); the first
 * part runs the forward ring, the second part runs the mirrored ring, each
 * with its own chunk_bounds(len, p).  Same arguments as the simulator, but
 * always the whole all-reduce (or only reduce-scatter if rs_only != 0). */
int orc_ring_simulate_bidir(void *const *bufs, int p, int64_t n, int dtype,
                            int op, int rs_only, int64_t *sends);

/* Closed-form per-element fold, for sampled checks on large inputs.
 *   vals   p * m elements: vals[r * m + j] is rank r's input at index idx[j]
 *   idx    m element indices in [0, n)
 *   mode   0 forward ring, 1 bidirectional, 2 tree order (see orc_tree_fold)
 *   out    m elements, the all-reduced value at each sampled index
 * Returns 0, or -1 on bad arguments. */
int orc_fold_sampled(const void *vals, const int64_t *idx, int64_t m, int p,
                     int64_t n, int dtype, int op, int mode, void *out);

/* Tree order: per element, adjacent pairs (x0 + x1, x2 + x3, ...) are
 * combined level by level, an odd last entry is carried to the next level
 * unchanged, and every combine rounds to the dtype.  bufs as in the
 * simulator, in place. */
int orc_tree_fold(void *const *bufs, int p, int64_t n, int dtype, int op);

/* Hierarchical 2D all-reduce ("Ring All-Reduce, in depth", "What real
 * libraries add" paragraph "Hierarchy", and "Worked example: flat versus
 * hierarchical").  p = m * g ranks in m nodes of g; rank r = node * g + local.
 *   1. reduce-scatter inside every node: a ring over its g ranks on
 *      chunk_bounds(n, g); local rank l then holds its node's partial of
 *      chunk (l + 1) mod g (its 1/g shard);
 *   2. all-reduce of that shard across nodes, among the m ranks with the same
 *      local rank: a ring over the nodes on chunk_bounds(shard, m); for avg
 *      the owner scales by 1/p (p = all ranks) before this ring's all-gather;
 *   3. all-gather inside every node.
 * g == p is the flat ring; g == 1 is the flat ring run across the nodes.
 * sends_intra / sends_inter (nullable, p entries): elements each rank sent
 * within its node and across nodes.  Returns 0, or -1 on bad arguments
 * (g < 1 or g not dividing p). */
int orc_hier_simulate(void *const *bufs, int p, int g, int64_t n, int dtype,
                      int op, int64_t *sends_intra, int64_t *sends_inter);

/* Closed-form per-element fold of the hierarchical schedule, as
 * orc_fold_sampled: element i of intra-node chunk c and shard sub-chunk s is
 * sum over nodes s, s+1, ... (mod m) of each node's partial, the partial
 * summing local ranks c, c+1, ... (mod g) of that node. */
int orc_hier_fold_sampled(const void *vals, const int64_t *idx, int64_t m_samples,
                          int p, int g, int64_t n, int dtype, int op, void *out);

/* fp64 reference for float inputs: ref[i] = sum_r x_r[i] and
 * mag[i] = sum_r |x_r[i]| in double.  Inputs are f32/bf16/f16. */
int orc_f64_sum(const void *const *bufs, int p, int64_t n, int dtype,
                double *ref, double *mag);

#ifdef __cplusplus
}
#endif
#endif
