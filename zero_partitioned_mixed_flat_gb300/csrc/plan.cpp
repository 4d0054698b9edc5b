// plan.cpp -- host side of libzero: the flat-buffer partitioner, the
// accounting, argument validation, the per-step state machine and the
// extern "C" entry points declared in include/zero.h.
#include "zero.h"
#include "zero_internal.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

namespace {

thread_local std::string g_last_error;

zero_status fail(zero_status code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

zero_status cuda_fail(cudaError_t e, const char *what) {
    return fail(ZERO_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t round_up(int64_t x, int64_t q) { return q == 0 ? x : ((x + q - 1) / q) * q; }

enum Phase { kIdle = 0, kReducing = 1, kDecided = 2 };


}  // namespace

namespace zk {
void set_last_error(const char *msg) { g_last_error = msg ? msg : ""; }
}  // namespace zk

static_assert(zk::kTile == ZERO_NORM_TILE, "the header's norm tile is the kernels' tile");

struct zero_plan {
    // layout
    int64_t psi = 0, psi_p = 0, part = 0;
    int32_t n_ranks = 1, align = 128, stage = 1, lp = 0;
    std::vector<int64_t> sizes, tensor_off;
    std::vector<int32_t> unit_of;
    std::vector<int64_t> unit_off, unit_pad;  // unit_off has n_units + 1 entries
    int64_t tiles_per_part = 0;
    // norm tiles restart at every unit's shard (one unit unless stage 3), so a
    // unit reduced alone gives the same bits as the whole partition
    std::vector<int64_t> unit_tile_base;  // first tile of each unit's shard
    std::vector<int64_t> unit_part_off;   // each unit's shard offset in the partition
    int32_t slots = 1;  // partition slots with partial sums (N, or 1 for DDP)
    // device scratch (allocated on first device call)
    int device = -1;
    double *d_partials = nullptr;
    double *d_level2 = nullptr;   // chunk sums of the partials (decision)
    double *d_level2x = nullptr;  // the same for the statistics export
    unsigned *d_overflow = nullptr;  // one overflow word per partition slot
    zk::StepRecord *d_rec = nullptr;
    cudaStream_t io = nullptr;  // private non-blocking stream for record reads/writes
    // completion of the plan's own device work: one event per stream used
    // since the last synchronising call
    std::vector<std::pair<cudaStream_t, cudaEvent_t>> pending;
    std::vector<cudaEvent_t> spare_events;
    bool captured = false;  // some call was enqueued on a capturing stream
    // step state (host)
    Phase phase = kIdle;
    uint64_t active[ZERO_MAX_RANKS / 64] = {0};
    int32_t growth_interval = 1000;
    int32_t reduce_lp_accum = 0;  // 1: partial sums rounded to the lp type
    int32_t quant_format = ZERO_QUANT_INT8;  // codes of the quantized gather
    int64_t spin_limit = zk::kDefaultSpinLimit;
    // the device step counter as far as the host can tell without reading it:
    // the last value read back or set, plus one per decision launched since
    int64_t t_hint = 0;
    bool use_global = false;  // zero_step_set_global_stats was called this step
    const double *global_stats = nullptr;  // device address of the caller's vector

    int32_t n_units() const { return int32_t(unit_pad.size()); }
    int64_t shard_len(int32_t u) const { return stage == 0 ? unit_pad[u] : unit_pad[u] / n_ranks; }
};

namespace {

// Build the layout.  The flat buffer is the tensors back to back; every unit
// (one unit unless stage 3) is padded up to a multiple of n_ranks * align.
zero_status build_layout(zero_plan *p) {
    const int64_t quantum = int64_t(p->n_ranks) * p->align;
    const size_t nt = p->sizes.size();
    p->tensor_off.assign(nt, 0);
    p->unit_off.clear();
    p->unit_pad.clear();
    int64_t flat = 0, total = 0;
    size_t t = 0;
    int32_t unit = 0;
    do {
        int64_t fill = 0;
        p->unit_off.push_back(flat);
        while (t < nt && (p->unit_of.empty() || p->unit_of[t] == unit)) {
            p->tensor_off[t] = flat + fill;
            fill += p->sizes[t];
            ++t;
        }
        const int64_t padded = round_up(fill, quantum);
        p->unit_pad.push_back(padded);
        flat += padded;
        total += fill;
        ++unit;
    } while (t < nt);
    p->unit_off.push_back(flat);
    p->psi = total;
    p->psi_p = flat;
    p->part = p->stage == 0 ? flat : flat / p->n_ranks;
    p->slots = p->stage == 0 ? 1 : p->n_ranks;
    p->unit_tile_base.assign(p->unit_pad.size(), 0);
    p->unit_part_off.assign(p->unit_pad.size(), 0);
    int64_t tiles = 0, off = 0;
    for (size_t u = 0; u < p->unit_pad.size(); ++u) {
        p->unit_tile_base[u] = tiles;
        p->unit_part_off[u] = off;
        const int64_t shard = p->shard_len(int32_t(u));
        tiles += (shard + zk::kTile - 1) / zk::kTile;
        off += shard;
    }
    p->tiles_per_part = tiles;
    return ZERO_OK;
}

void free_scratch(zero_plan *p) {
    cudaFree(p->d_partials);
    cudaFree(p->d_level2);
    cudaFree(p->d_level2x);
    cudaFree(p->d_overflow);
    cudaFree(p->d_rec);
    p->d_partials = p->d_level2 = p->d_level2x = nullptr;
    p->d_overflow = nullptr;
    p->d_rec = nullptr;
    if (p->io) cudaStreamDestroy(p->io);
    p->io = nullptr;
}

zero_status ensure_device(zero_plan *p) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (p->device >= 0) {
        if (dev != p->device)
            return fail(ZERO_EINVAL, "plan scratch lives on device %d, current device is %d", p->device,
                        dev);
        return ZERO_OK;
    }
    const size_t n_part = size_t(p->slots) * size_t(p->tiles_per_part > 0 ? p->tiles_per_part : 1);
    const size_t n_level2 = size_t(p->slots) *
                            size_t(std::max<int64_t>(1, (p->tiles_per_part + zk::kPartialChunk - 1) / zk::kPartialChunk));
    bool ok = cudaMalloc(reinterpret_cast<void **>(&p->d_partials), n_part * sizeof(double)) == cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void **>(&p->d_level2), n_level2 * sizeof(double)) == cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void **>(&p->d_level2x), n_level2 * sizeof(double)) == cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void **>(&p->d_overflow), size_t(p->slots) * sizeof(unsigned)) ==
                   cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void **>(&p->d_rec), sizeof(zk::StepRecord)) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        free_scratch(p);
        return fail(ZERO_ENOMEM, "cudaMalloc of the plan scratch (%zu partial sums) failed", n_part);
    }
    e = cudaStreamCreateWithFlags(&p->io, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        p->io = nullptr;
        free_scratch(p);
        return cuda_fail(e, "cudaStreamCreateWithFlags");
    }
    zk::StepRecord init;
    std::memset(&init, 0, sizeof init);
    init.coef = 1.0f;
    e = cudaMemcpyAsync(p->d_rec, &init, sizeof init, cudaMemcpyHostToDevice, p->io);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->d_partials, 0, n_part * sizeof(double), p->io);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->d_overflow, 0, size_t(p->slots) * sizeof(unsigned), p->io);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->io);
    if (e != cudaSuccess) {
        free_scratch(p);
        return cuda_fail(e, "initialising the plan scratch");
    }
    p->device = dev;
    return ZERO_OK;
}

// Remember that the plan's device work was enqueued on stream s (called after
// a call's launches succeeded).  A capturing stream records nothing: the graph
// may be replayed anywhere, so the plan then waits for the whole device.
zero_status note_work(zero_plan *p, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        cs = cudaStreamCaptureStatusActive;
    }
    if (cs != cudaStreamCaptureStatusNone) {
        p->captured = true;
        return ZERO_OK;
    }
    cudaEvent_t ev = nullptr;
    for (auto &pe : p->pending)
        if (pe.first == s) ev = pe.second;
    if (!ev) {
        if (!p->spare_events.empty()) {
            ev = p->spare_events.back();
            p->spare_events.pop_back();
        } else {
            cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreateWithFlags");
        }
        p->pending.emplace_back(s, ev);
    }
    cudaError_t e = cudaEventRecord(ev, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    return ZERO_OK;
}

// Wait for the plan's own device work: the events of the streams it used since
// the last wait (or the whole device if a call was captured into a graph).
zero_status wait_own_work(zero_plan *p) {
    cudaError_t err = cudaSuccess;
    if (p->captured) {
        err = cudaDeviceSynchronize();
    } else {
        for (auto &pe : p->pending) {
            cudaError_t e = cudaEventSynchronize(pe.second);
            if (err == cudaSuccess) err = e;
        }
    }
    for (auto &pe : p->pending) p->spare_events.push_back(pe.second);
    p->pending.clear();
    if (err != cudaSuccess) return cuda_fail(err, p->captured ? "cudaDeviceSynchronize" : "cudaEventSynchronize");
    return ZERO_OK;
}

// Where the device can read an input buffer from: its own memory, managed
// memory, pinned host memory (through the pinned buffer's device address;
// over NVLink-C2C on Grace systems), or pageable host memory when the device
// reads the host page tables.  Anything else is refused before any launch.
zero_status readable_by_device(const void *ptr, int dev, const char *what, int32_t j,
                               const void **out) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(ZERO_EINVAL, "%s[%d]: cudaPointerGetAttributes: %s", what, j, cudaGetErrorString(e));
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
        if (a.device != dev)
            return fail(ZERO_EINVAL, "%s[%d] lives on device %d, the current device is %d", what, j,
                        a.device, dev);
        *out = ptr;
        return ZERO_OK;
    case cudaMemoryTypeManaged:
        *out = ptr;
        return ZERO_OK;
    case cudaMemoryTypeHost:
        if (!a.devicePointer) return fail(ZERO_EINVAL, "%s[%d]: pinned host memory without a device mapping", what, j);
        if (!aligned16(a.devicePointer)) return fail(ZERO_EALIGN, "%s[%d]: device mapping not 16-byte aligned", what, j);
        *out = a.devicePointer;
        return ZERO_OK;
    default: {
        int pageable = 0;
        if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) {
            cudaGetLastError();
            pageable = 0;
        }
        if (!pageable)
            return fail(ZERO_EINVAL, "%s[%d] is pageable host memory this device cannot read; pin it", what, j);
        *out = ptr;
        return ZERO_OK;
    }
    }
}

zero_status check_rank(const zero_plan *p, int32_t rank) {
    if (rank < 0 || rank >= p->n_ranks) return fail(ZERO_EINVAL, "rank %d outside [0, %d)", rank, p->n_ranks);
    if (p->stage == 0 && rank != 0)
        return fail(ZERO_EINVAL, "stage 0 (DDP) simulates one replica: rank must be 0");
    return ZERO_OK;
}

}  // namespace

extern "C" {

const char *zero_last_error(void) { return g_last_error.c_str(); }

zero_status zero_plan_create(int64_t psi, int32_t n_ranks, const int64_t *tensor_sizes,
                             int32_t n_tensors, int32_t align, int32_t stage,
                             const int32_t *unit_of_tensor, zero_lp lp, zero_plan **out) {
    if (!out) return fail(ZERO_EINVAL, "out is NULL");
    *out = nullptr;
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS)
        return fail(ZERO_EINVAL, "n_ranks %d outside [1, %d]", n_ranks, ZERO_MAX_RANKS);
    if (align < 8 || align % 8 != 0) return fail(ZERO_EINVAL, "align %d is not a positive multiple of 8", align);
    if (stage < 0 || stage > 3) return fail(ZERO_EINVAL, "stage %d outside [0, 3]", stage);
    if (lp != ZERO_FP16 && lp != ZERO_BF16) return fail(ZERO_EINVAL, "unknown lp type %d", int(lp));
    if (n_tensors < 0) return fail(ZERO_EINVAL, "n_tensors < 0");
    if (n_tensors > 0 && !tensor_sizes) return fail(ZERO_EINVAL, "tensor_sizes is NULL");
    zero_plan *p = new (std::nothrow) zero_plan();
    if (!p) return fail(ZERO_ENOMEM, "host allocation of the plan failed");
    p->n_ranks = n_ranks;
    p->align = align;
    p->stage = stage;
    p->lp = lp;
    if (n_tensors == 0 || !tensor_sizes) {
        if (psi < 0) {
            delete p;
            return fail(ZERO_EINVAL, "psi < 0 without a tensor list");
        }
        p->sizes.assign(1, psi);
    } else {
        int64_t sum = 0;
        p->sizes.assign(tensor_sizes, tensor_sizes + n_tensors);
        for (int64_t s : p->sizes) {
            if (s < 0) {
                delete p;
                return fail(ZERO_EINVAL, "negative tensor size");
            }
            sum += s;
        }
        if (psi >= 0 && psi != sum) {
            delete p;
            return fail(ZERO_EINVAL, "psi %lld differs from the tensor sizes' sum %lld", (long long)psi,
                        (long long)sum);
        }
    }
    if (stage == 3 && unit_of_tensor && n_tensors > 0) {
        p->unit_of.assign(unit_of_tensor, unit_of_tensor + n_tensors);
        if (p->unit_of[0] != 0) {
            delete p;
            return fail(ZERO_EINVAL, "unit_of_tensor must start at unit 0");
        }
        for (int32_t t = 1; t < n_tensors; ++t) {
            const int32_t d = p->unit_of[t] - p->unit_of[t - 1];
            if (d != 0 && d != 1) {
                delete p;
                return fail(ZERO_EINVAL, "unit_of_tensor must be non-decreasing without gaps");
            }
        }
    }
    build_layout(p);
    *out = p;
    return ZERO_OK;
}

zero_status zero_plan_query(const zero_plan *p, int64_t *psi_padded, int64_t *part_len,
                            int64_t *tensor_offsets) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (psi_padded) *psi_padded = p->psi_p;
    if (part_len) *part_len = p->part;
    if (tensor_offsets)
        std::memcpy(tensor_offsets, p->tensor_off.data(), p->tensor_off.size() * sizeof(int64_t));
    return ZERO_OK;
}

zero_status zero_plan_units(const zero_plan *p, int32_t *n_units, int64_t *unit_offsets,
                            int64_t *unit_padded) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (n_units) *n_units = p->n_units();
    if (unit_offsets) std::memcpy(unit_offsets, p->unit_off.data(), p->unit_off.size() * sizeof(int64_t));
    if (unit_padded) std::memcpy(unit_padded, p->unit_pad.data(), p->unit_pad.size() * sizeof(int64_t));
    return ZERO_OK;
}

zero_status zero_plan_unit_shards(const zero_plan *p, int64_t *shard_len, int64_t *shard_offset) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    for (int32_t u = 0; u < p->n_units(); ++u) {
        if (shard_len) shard_len[u] = p->shard_len(u);
        if (shard_offset) shard_offset[u] = p->unit_part_off[size_t(u)];
    }
    return ZERO_OK;
}

zero_status zero_plan_fragments(const zero_plan *p, int32_t rank, int64_t max_frag, int64_t *frag,
                                int64_t *count) {
    if (!p || !count) return fail(ZERO_EINVAL, "plan or count is NULL");
    if (rank < 0 || rank >= p->n_ranks) return fail(ZERO_EINVAL, "rank %d outside [0, %d)", rank, p->n_ranks);
    if (max_frag > 0 && !frag) return fail(ZERO_EINVAL, "frag is NULL");
    int64_t n = 0, part_pos = 0;
    size_t t = 0;
    for (int32_t u = 0; u < p->n_units(); ++u) {
        const int64_t shard = p->shard_len(u);
        const int64_t lo = p->unit_off[u] + (p->stage == 0 ? 0 : rank * shard);
        const int64_t hi = lo + shard;
        // tensors of unit u are contiguous in the list
        for (; t < p->sizes.size() && (p->unit_of.empty() || p->unit_of[t] == u); ++t) {
            const int64_t a = std::max(lo, p->tensor_off[t]);
            const int64_t b = std::min(hi, p->tensor_off[t] + p->sizes[t]);
            if (a >= b) continue;
            if (n < max_frag) {
                frag[4 * n + 0] = int64_t(t);
                frag[4 * n + 1] = a - p->tensor_off[t];
                frag[4 * n + 2] = part_pos + (a - lo);
                frag[4 * n + 3] = b - a;
            }
            ++n;
        }
        part_pos += shard;
    }
    *count = n;
    return ZERO_OK;
}

zero_status zero_plan_set_loss_scaler(zero_plan *p, int32_t growth_interval) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    p->growth_interval = growth_interval;
    return ZERO_OK;
}

zero_status zero_plan_set_reduce_precision(zero_plan *p, int32_t accumulate_in_lp) {
    if (!p || (accumulate_in_lp != 0 && accumulate_in_lp != 1))
        return fail(ZERO_EINVAL, "plan is NULL or accumulate_in_lp is not 0/1");
    p->reduce_lp_accum = accumulate_in_lp;
    return ZERO_OK;
}

zero_status zero_plan_set_gather_quantization(zero_plan *p, int32_t format) {
    if (!p || (format != ZERO_QUANT_INT8 && format != ZERO_QUANT_FP8_E4M3))
        return fail(ZERO_EINVAL, "plan is NULL or format is not ZERO_QUANT_INT8 / ZERO_QUANT_FP8_E4M3");
    p->quant_format = format;
    return ZERO_OK;
}

zero_status zero_plan_set_spin_limit(zero_plan *p, int64_t polls) {
    if (!p || polls < 0) return fail(ZERO_EINVAL, "plan is NULL or polls < 0");
    p->spin_limit = polls;
    return ZERO_OK;
}

zero_status zero_plan_set_state(zero_plan *p, int64_t step, int32_t good_steps) {
    if (!p || step < 0 || good_steps < 0) return fail(ZERO_EINVAL, "bad plan state");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    st = wait_own_work(p);
    if (st != ZERO_OK) return st;
    zk::StepRecord rec;
    cudaError_t e = cudaMemcpyAsync(&rec, p->d_rec, sizeof rec, cudaMemcpyDeviceToHost, p->io);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->io);
    if (e != cudaSuccess) return cuda_fail(e, "reading the step record");
    rec.step = step;
    rec.good_steps = good_steps;
    e = cudaMemcpyAsync(p->d_rec, &rec, sizeof rec, cudaMemcpyHostToDevice, p->io);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->io);
    if (e != cudaSuccess) return cuda_fail(e, "writing the step record");
    p->t_hint = step;
    return ZERO_OK;
}

}  // extern "C"

namespace {

// Argument checks of one partition's reduce inputs (host only, no CUDA call).
zero_status check_reduce_args(const zero_plan *p, int32_t rank, const void *const *grad_slices,
                              const float *grad_out) {
    zero_status st = check_rank(p, rank);
    if (st != ZERO_OK) return st;
    if (!grad_slices || (!grad_out && p->part > 0)) return fail(ZERO_EINVAL, "NULL slices or output");
    for (int32_t j = 0; j < p->n_ranks; ++j) {
        if (!grad_slices[j] && p->part > 0) return fail(ZERO_EINVAL, "grad_slices[%d] is NULL", j);
        if (!aligned16(grad_slices[j])) return fail(ZERO_EALIGN, "grad_slices[%d] is not 16-byte aligned", j);
    }
    if (!aligned16(grad_out)) return fail(ZERO_EALIGN, "grad_out is not 16-byte aligned");
    return ZERO_OK;
}

// The argument checks, then the classification of the slice pointers (a CUDA
// query): the N translated slice pointers go to *src.
zero_status check_reduce_job(zero_plan *p, int32_t rank, const void *const *grad_slices, float *grad_out,
                             std::vector<const void *> *src) {
    zero_status st = check_reduce_args(p, rank, grad_slices, grad_out);
    if (st != ZERO_OK) return st;
    st = ensure_device(p);
    if (st != ZERO_OK) return st;
    src->assign(size_t(p->n_ranks), nullptr);
    if (p->part > 0)
        for (int32_t j = 0; j < p->n_ranks; ++j) {
            st = readable_by_device(grad_slices[j], p->device, "grad_slices", j, &(*src)[size_t(j)]);
            if (st != ZERO_OK) return st;
        }
    return ZERO_OK;
}

zero_status check_reduce_scalars(float loss_scale, int64_t bucket_elems) {
    if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale))
        return fail(ZERO_EINVAL, "loss_scale must be finite and > 0");
    if (bucket_elems < 0) return fail(ZERO_EINVAL, "bucket_elems < 0");
    return ZERO_OK;
}

// On the first reduce of a step: forget the previous step's partitions,
// partial sums and overflow words (a partition reduced only in part then adds
// only that part).
zero_status start_step(zero_plan *p, cudaStream_t s) {
    if (p->phase == kReducing) return ZERO_OK;
    std::memset(p->active, 0, sizeof p->active);
    p->use_global = false;
    p->global_stats = nullptr;
    cudaError_t e = cudaMemsetAsync(p->d_overflow, 0, size_t(p->slots) * sizeof(unsigned), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(overflow)");
    if (p->tiles_per_part > 0) {
        e = cudaMemsetAsync(p->d_partials, 0, size_t(p->slots) * size_t(p->tiles_per_part) * sizeof(double), s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(partials)");
    }
    p->phase = kReducing;
    return ZERO_OK;
}

// One partition's reduce: units [first, first + count) of partition slot
// `slot` (one unit unless stage 3) from the N slices src into grad_out.
struct ReduceJob {
    int32_t slot;
    int32_t first, count;
    const void *const *src;
    float *grad_out;
};

// Reduce the jobs in order.  Each unit is cut into pieces of whole norm tiles
// counted from the unit's start (bucket_elems rounded up to tiles; 0 = the
// whole unit); consecutive pieces, of one partition or of several, share one
// kernel launch while their total stays within one bucket (any number when
// bucket_elems is 0), up to the kernel's segment and slice-table limits.  The
// grouping only decides launches: every tile's partial is the same.
zero_status reduce_jobs(zero_plan *p, const std::vector<ReduceJob> &jobs, float loss_scale,
                        int64_t bucket_elems, cudaStream_t s) {
    const float inv = float(1.0 / (double(loss_scale) * double(p->n_ranks)));
    const int64_t piece = bucket_elems == 0 ? 0 : round_up(bucket_elems, zk::kTile);
    const size_t table = size_t(zk::reduce_src_table(p->n_ranks));
    std::vector<const void *> srcs;
    std::vector<zk::ReduceSegment> segs;
    int64_t launch_elems = 0;
    int64_t in_table = -1;  // the job whose slices were appended last
    int32_t src0 = 0;
    auto flush = [&]() -> zero_status {
        if (segs.empty()) return ZERO_OK;
        cudaError_t e = zk::launch_reduce(srcs.data(), int(srcs.size()), p->n_ranks, p->lp, p->reduce_lp_accum,
                                          segs.data(), int(segs.size()), inv, s);
        segs.clear();
        srcs.clear();
        in_table = -1;
        launch_elems = 0;
        if (e != cudaSuccess) return cuda_fail(e, "reduce kernel launch");
        return ZERO_OK;
    };
    for (size_t ji = 0; ji < jobs.size(); ++ji) {
        const ReduceJob &jb = jobs[ji];
        double *partials = p->d_partials + int64_t(jb.slot) * p->tiles_per_part;
        for (int32_t u = jb.first; u < jb.first + jb.count; ++u) {
            const int64_t shard = p->shard_len(u);
            const int64_t base = p->unit_part_off[size_t(u)];
            const int64_t step = piece == 0 ? std::max<int64_t>(shard, 1) : piece;
            for (int64_t b0 = 0; b0 < shard; b0 += step) {
                const int64_t len = std::min(step, shard - b0);
                const size_t need = in_table == int64_t(ji) ? 0 : size_t(p->n_ranks);
                if (!segs.empty() && ((piece > 0 && launch_elems + len > piece) ||
                                      int(segs.size()) == zk::kMaxReduceSegments || srcs.size() + need > table)) {
                    zero_status st = flush();
                    if (st != ZERO_OK) return st;
                }
                if (in_table != int64_t(ji)) {
                    src0 = int32_t(srcs.size());
                    srcs.insert(srcs.end(), jb.src, jb.src + p->n_ranks);
                    in_table = int64_t(ji);
                }
                segs.push_back({base + b0, len, p->unit_tile_base[size_t(u)] + b0 / zk::kTile, jb.grad_out, partials,
                                p->d_overflow + jb.slot, src0});
                launch_elems += len;
            }
        }
    }
    return flush();
}

}  // namespace

extern "C" {

zero_status zero_reduce_partition(zero_plan *p, int32_t rank, const void *const *grad_slices,
                                  float *grad_out, float loss_scale, int64_t bucket_elems,
                                  void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    zero_status st = check_reduce_scalars(loss_scale, bucket_elems);
    if (st != ZERO_OK) return st;
    std::vector<const void *> src;
    st = check_reduce_job(p, rank, grad_slices, grad_out, &src);
    if (st != ZERO_OK) return st;
    st = start_step(p, s);
    if (st != ZERO_OK) return st;
    const int32_t slot = p->stage == 0 ? 0 : rank;
    p->active[slot >> 6] |= uint64_t(1) << (slot & 63);
    st = reduce_jobs(p, {ReduceJob{slot, 0, p->n_units(), src.data(), grad_out}}, loss_scale, bucket_elems, s);
    if (st != ZERO_OK) return st;
    return note_work(p, s);
}

zero_status zero_reduce_partitions(zero_plan *p, int32_t n_parts, const int32_t *ranks,
                                   const void *const *grad_slices, float *const *grad_out,
                                   float loss_scale, int64_t bucket_elems, void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (n_parts < 1 || n_parts > p->n_ranks || !ranks || !grad_slices || !grad_out)
        return fail(ZERO_EINVAL, "n_parts outside [1, N] or a NULL array");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    zero_status st = check_reduce_scalars(loss_scale, bucket_elems);
    if (st != ZERO_OK) return st;
    std::vector<char> seen(size_t(p->n_ranks), 0);
    for (int32_t i = 0; i < n_parts; ++i) {  // every argument before any CUDA call
        st = check_reduce_args(p, ranks[i], grad_slices + int64_t(i) * p->n_ranks, grad_out[i]);
        if (st != ZERO_OK) return st;
        if (seen[size_t(ranks[i])]++) return fail(ZERO_EINVAL, "rank %d listed twice", ranks[i]);
    }
    std::vector<std::vector<const void *>> srcs(static_cast<size_t>(n_parts));
    std::vector<ReduceJob> jobs;
    for (int32_t i = 0; i < n_parts; ++i) {
        st = check_reduce_job(p, ranks[i], grad_slices + int64_t(i) * p->n_ranks, grad_out[i], &srcs[size_t(i)]);
        if (st != ZERO_OK) return st;
        jobs.push_back({p->stage == 0 ? 0 : ranks[i], 0, p->n_units(), srcs[size_t(i)].data(), grad_out[i]});
    }
    st = start_step(p, s);
    if (st != ZERO_OK) return st;
    for (const ReduceJob &jb : jobs) p->active[jb.slot >> 6] |= uint64_t(1) << (jb.slot & 63);
    st = reduce_jobs(p, jobs, loss_scale, bucket_elems, s);
    if (st != ZERO_OK) return st;
    return note_work(p, s);
}

zero_status zero_reduce_units(zero_plan *p, int32_t rank, int32_t first_unit, int32_t n_units,
                              const void *const *grad_slices, float *grad_out, float loss_scale,
                              void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (p->stage != 3) return fail(ZERO_EINVAL, "zero_reduce_units needs a stage-3 plan");
    if (first_unit < 0 || n_units < 1 || first_unit + n_units > p->n_units())
        return fail(ZERO_EINVAL, "units [%d, %d) outside [0, %d)", first_unit, first_unit + n_units,
                    p->n_units());
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    zero_status st = check_reduce_scalars(loss_scale, 0);
    if (st != ZERO_OK) return st;
    std::vector<const void *> src;
    st = check_reduce_job(p, rank, grad_slices, grad_out, &src);
    if (st != ZERO_OK) return st;
    st = start_step(p, s);
    if (st != ZERO_OK) return st;
    p->active[rank >> 6] |= uint64_t(1) << (rank & 63);
    st = reduce_jobs(p, {ReduceJob{rank, first_unit, n_units, src.data(), grad_out}}, loss_scale, 0, s);
    if (st != ZERO_OK) return st;
    return note_work(p, s);
}

zero_status zero_partition_stats(zero_plan *p, double *stats, void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (!stats) return fail(ZERO_EINVAL, "stats is NULL");
    if (reinterpret_cast<uintptr_t>(stats) & 7u) return fail(ZERO_EALIGN, "stats is not 8-byte aligned");
    if (p->phase != kReducing) return fail(ZERO_ESTATE, "no partition reduced in the current step");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    const void *dst = nullptr;
    st = readable_by_device(stats, p->device, "stats", 0, &dst);
    if (st != ZERO_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    zk::NormLaunch a = {};
    a.mode = zk::kExportStats;
    a.partials = p->d_partials;
    a.level2 = p->d_level2x;
    a.arrivals = &p->d_rec->arrivals_x;
    a.overflow = p->d_overflow;
    a.stats_out = static_cast<double *>(const_cast<void *>(dst));
    a.tiles_per_slot = p->tiles_per_part;
    a.active_mask = p->active;
    a.n_slots = p->n_ranks;
    a.rec = p->d_rec;
    cudaError_t e = zk::launch_norm(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "statistics kernel launch");
    return note_work(p, s);
}

zero_status zero_step_set_global_stats(zero_plan *p, const double *stats) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (!stats) return fail(ZERO_EINVAL, "stats is NULL");
    if (reinterpret_cast<uintptr_t>(stats) & 7u) return fail(ZERO_EALIGN, "stats is not 8-byte aligned");
    if (p->phase != kReducing)
        return fail(ZERO_ESTATE, "global stats belong between a step's reduces and its first Adam call");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    const void *src = nullptr;
    st = readable_by_device(stats, p->device, "stats", 0, &src);
    if (st != ZERO_OK) return st;
    p->use_global = true;
    p->global_stats = static_cast<const double *>(src);
    return ZERO_OK;
}

}  // extern "C"

namespace {

// One partition's part of an Adam call: elements [begin, begin + len) of
// rank `rank`'s partition, with that call's pointers.
struct AdamJob {
    int32_t rank;
    int64_t begin, len;
    const float *grad;
    float *master, *m, *v;
    void *param_out;
};

zero_status check_adam_job(const zero_plan *p, const AdamJob &j) {
    zero_status st = check_rank(p, j.rank);
    if (st != ZERO_OK) return st;
    if (p->part > 0 && (!j.grad || !j.master || !j.m || !j.v)) return fail(ZERO_EINVAL, "NULL state pointer");
    if (!aligned16(j.grad) || !aligned16(j.master) || !aligned16(j.m) || !aligned16(j.v) || !aligned16(j.param_out))
        return fail(ZERO_EALIGN, "a state or parameter pointer is not 16-byte aligned");
    return ZERO_OK;
}

// The decision (first call of a step) and the Adam launches over the jobs,
// shared by zero_adam_step (one whole partition), zero_adam_step_range (one
// sub-group) and zero_adam_step_partitions (several partitions, one launch
// per kMaxAdamSegments of them).
zero_status adam_impl(zero_plan *p, const std::vector<AdamJob> &jobs, float lr, float beta1,
                      float beta2, float eps, float wd, int32_t adamw, float loss_scale, float clip,
                      double remote_sumsq, int32_t remote_overflow, void *stream) {
    for (const AdamJob &j : jobs) {
        zero_status st = check_adam_job(p, j);
        if (st != ZERO_OK) return st;
    }
    if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale))
        return fail(ZERO_EINVAL, "loss_scale must be finite and > 0");
    if (!(remote_sumsq >= 0.0)) return fail(ZERO_EINVAL, "remote_sumsq must be >= 0");
    if (p->phase == kIdle) return fail(ZERO_ESTATE, "zero_adam_step before any zero_reduce_partition");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->phase == kReducing) {
        bool any = false;
        for (uint64_t w : p->active) any = any || w != 0;
        if (!any) return fail(ZERO_ESTATE, "no partition was reduced in the current step");
        // bias corrections, computed as the oracle does, for the counters
        // t_hint + 1 down to t_hint + 2 - kBcTable (t_hint + 1 unless earlier
        // steps were skipped since the counter was last read back)
        const int64_t bc_t0 = p->t_hint + 1;
        float bc1[zk::kBcTable], bc2[zk::kBcTable];
        for (int i = 0; i < zk::kBcTable; ++i) {
            const int64_t t = bc_t0 - i;
            bc1[i] = t > 0 ? float(1.0 - std::pow(double(beta1), double(t))) : 0.0f;
            bc2[i] = t > 0 ? float(1.0 - std::pow(double(beta2), double(t))) : 0.0f;
        }
        zk::NormLaunch a = {};
        a.mode = p->use_global ? zk::kDecideGlobal : zk::kDecideLocal;
        a.partials = p->d_partials;
        a.level2 = p->d_level2;
        a.arrivals = &p->d_rec->arrivals;
        a.overflow = p->d_overflow;
        a.stats_in = p->global_stats;
        a.tiles_per_slot = p->tiles_per_part;
        a.active_mask = p->active;
        a.n_slots = p->n_ranks;
        a.remote_sumsq = remote_sumsq;
        a.remote_overflow = remote_overflow ? 1 : 0;
        a.clip = clip;
        a.loss_scale = loss_scale;
        a.beta1 = beta1;
        a.beta2 = beta2;
        a.growth_interval = p->growth_interval;
        a.bc_t0 = bc_t0;
        a.bc1_tab = bc1;
        a.bc2_tab = bc2;
        a.rec = p->d_rec;
        cudaError_t e = zk::launch_norm(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "decide kernel launch");
        p->phase = kDecided;
        p->t_hint += 1;
    }
    const float omb1 = 1.0f - beta1;
    const float omb2 = 1.0f - beta2;
    const float decay = float(1.0 - double(lr) * double(wd));
    std::vector<zk::AdamSegment> segs;
    auto flush = [&]() -> zero_status {
        if (segs.empty()) return ZERO_OK;
        cudaError_t e = zk::launch_adam(segs.data(), int(segs.size()), p->lp, p->d_rec, &p->d_rec->error,
                                        p->spin_limit, lr, beta1, beta2, omb1, omb2, eps, wd, decay,
                                        adamw ? 1 : 0, s);
        segs.clear();
        if (e != cudaSuccess) return cuda_fail(e, "adam kernel launch");
        return ZERO_OK;
    };
    for (const AdamJob &j : jobs) {
        if (j.len == 0) continue;
        void *param = nullptr;
        if (j.param_out) {
            const int64_t off = ((p->stage == 3) ? 0 : int64_t(j.rank) * p->part) + j.begin;
            param = static_cast<uint16_t *>(j.param_out) + off;
        }
        segs.push_back({j.grad + j.begin, j.master + j.begin, j.m + j.begin, j.v + j.begin, param, j.len});
        if (int(segs.size()) == zk::kMaxAdamSegments) {
            st = flush();
            if (st != ZERO_OK) return st;
        }
    }
    st = flush();
    if (st != ZERO_OK) return st;
    return note_work(p, s);
}

}  // namespace

extern "C" {

zero_status zero_adam_step(zero_plan *p, int32_t rank, const float *grad, float *master, float *m,
                           float *v, void *param_out, float lr, float beta1, float beta2, float eps,
                           float wd, int32_t adamw, float loss_scale, float clip,
                           double remote_sumsq, int32_t remote_overflow, void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    return adam_impl(p, {AdamJob{rank, 0, p->part, grad, master, m, v, param_out}}, lr, beta1, beta2, eps, wd,
                     adamw, loss_scale, clip, remote_sumsq, remote_overflow, stream);
}

zero_status zero_adam_step_range(zero_plan *p, int32_t rank, int64_t begin, int64_t len,
                                 const float *grad, float *master, float *m, float *v,
                                 void *param_out, float lr, float beta1, float beta2, float eps,
                                 float wd, int32_t adamw, float loss_scale, float clip,
                                 double remote_sumsq, int32_t remote_overflow, void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (begin < 0 || len < 0 || begin > p->part || len > p->part - begin)
        return fail(ZERO_EINVAL, "range [%lld, %lld + %lld) outside the partition of %lld elements",
                    (long long)begin, (long long)begin, (long long)len, (long long)p->part);
    if (begin % 8 != 0 || len % 8 != 0)
        return fail(ZERO_EALIGN, "sub-group begin and length must be multiples of 8 elements");
    return adam_impl(p, {AdamJob{rank, begin, len, grad, master, m, v, param_out}}, lr, beta1, beta2, eps, wd,
                     adamw, loss_scale, clip, remote_sumsq, remote_overflow, stream);
}

zero_status zero_adam_step_partitions(zero_plan *p, int32_t n_parts, const int32_t *ranks,
                                      const float *const *grad, float *const *master, float *const *m,
                                      float *const *v, void *const *param_out, float lr, float beta1,
                                      float beta2, float eps, float wd, int32_t adamw, float loss_scale,
                                      float clip, double remote_sumsq, int32_t remote_overflow,
                                      void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (n_parts < 1 || n_parts > p->n_ranks || !ranks || !grad || !master || !m || !v || !param_out)
        return fail(ZERO_EINVAL, "n_parts outside [1, N] or a NULL array");
    std::vector<AdamJob> jobs;
    std::vector<char> seen(size_t(p->n_ranks), 0);
    for (int32_t i = 0; i < n_parts; ++i) {
        if (ranks[i] < 0 || ranks[i] >= p->n_ranks)
            return fail(ZERO_EINVAL, "rank %d outside [0, %d)", ranks[i], p->n_ranks);
        if (seen[size_t(ranks[i])]++) return fail(ZERO_EINVAL, "rank %d listed twice", ranks[i]);
        jobs.push_back({ranks[i], 0, p->part, grad[i], master[i], m[i], v[i], param_out[i]});
    }
    return adam_impl(p, jobs, lr, beta1, beta2, eps, wd, adamw, loss_scale, clip, remote_sumsq,
                     remote_overflow, stream);
}

zero_status zero_step_result(zero_plan *p, double *norm, int32_t *skipped, float *new_loss_scale,
                             int64_t *step) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    st = wait_own_work(p);
    if (st != ZERO_OK) return st;
    zk::StepRecord rec;
    cudaError_t e = cudaMemcpyAsync(&rec, p->d_rec, sizeof rec, cudaMemcpyDeviceToHost, p->io);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->io);
    if (e != cudaSuccess) return cuda_fail(e, "reading the step record");
    p->t_hint = rec.step;
    if (norm) *norm = rec.norm;
    if (skipped) *skipped = rec.skip;
    if (new_loss_scale) *new_loss_scale = rec.loss_scale;
    if (step) *step = rec.step;
    if (rec.error) {
        e = cudaMemsetAsync(&p->d_rec->error, 0, sizeof(int), p->io);
        if (e == cudaSuccess) e = cudaStreamSynchronize(p->io);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the error word");
        return fail(ZERO_ETIMEOUT, "a bounded device wait gave up");
    }
    return ZERO_OK;
}

zero_status zero_plan_check(zero_plan *p) {
    return zero_step_result(p, nullptr, nullptr, nullptr, nullptr);
}

zero_status zero_gather_layer(zero_plan *p, int32_t unit, const void *const *shards, void *out,
                              void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (p->stage != 3) return fail(ZERO_EINVAL, "zero_gather_layer needs a stage-3 plan");
    if (unit < 0 || unit >= p->n_units()) return fail(ZERO_EINVAL, "unit %d outside [0, %d)", unit, p->n_units());
    const int64_t shard = p->shard_len(unit);
    if (!shards || (!out && shard > 0)) return fail(ZERO_EINVAL, "NULL shards or output");
    for (int32_t j = 0; j < p->n_ranks; ++j) {
        if (!shards[j] && shard > 0) return fail(ZERO_EINVAL, "shards[%d] is NULL", j);
        if (!aligned16(shards[j])) return fail(ZERO_EALIGN, "shards[%d] is not 16-byte aligned", j);
    }
    if (!aligned16(out)) return fail(ZERO_EALIGN, "out is not 16-byte aligned");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    int64_t off = 0;  // the unit's shard offset inside each rank's partition
    for (int32_t u = 0; u < unit; ++u) off += p->shard_len(u);
    cudaError_t e = zk::launch_gather(shards, p->n_ranks, off * 2, shard * 2, out, shard * 2, p->spin_limit,
                                      &p->d_rec->error, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
    return note_work(p, static_cast<cudaStream_t>(stream));
}

zero_status zero_allgather_params(zero_plan *p, const void *const *partitions, void *out,
                                  int64_t bucket_elems, void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (p->stage != 1 && p->stage != 2) return fail(ZERO_EINVAL, "zero_allgather_params needs a stage-1 or 2 plan");
    if (!partitions || (!out && p->part > 0)) return fail(ZERO_EINVAL, "NULL partitions or output");
    for (int32_t j = 0; j < p->n_ranks; ++j) {
        if (!partitions[j] && p->part > 0) return fail(ZERO_EINVAL, "partitions[%d] is NULL", j);
        if (!aligned16(partitions[j])) return fail(ZERO_EALIGN, "partitions[%d] is not 16-byte aligned", j);
    }
    if (!aligned16(out)) return fail(ZERO_EALIGN, "out is not 16-byte aligned");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    // per-rank run of one bucket: bucket_elems / N, a multiple of 8, at least 8
    int64_t run = p->part;
    if (bucket_elems > 0) {
        run = bucket_elems / p->n_ranks / 8 * 8;
        if (run < 8) run = 8;
    }
    for (int64_t k0 = 0; k0 < p->part; k0 += run) {
        const int64_t len = std::min(run, p->part - k0);
        cudaError_t e = zk::launch_gather(partitions, p->n_ranks, k0 * 2, len * 2,
                                          static_cast<uint16_t *>(out) + k0, p->part * 2, p->spin_limit,
                                          &p->d_rec->error, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
    }
    return note_work(p, static_cast<cudaStream_t>(stream));
}

zero_status zero_quantize_shard(zero_plan *p, const void *shard, int8_t *codes, float *scales,
                                void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (p->stage != 3) return fail(ZERO_EINVAL, "the quantized gather needs a stage-3 plan");
    if (p->align % ZERO_QUANT_BLOCK != 0)
        return fail(ZERO_EINVAL, "the quantized gather needs align to be a multiple of %d", ZERO_QUANT_BLOCK);
    if (p->part > 0 && (!shard || !codes || !scales)) return fail(ZERO_EINVAL, "NULL pointer argument");
    if (!aligned16(shard) || !aligned16(codes) || !aligned16(scales))
        return fail(ZERO_EALIGN, "shard, codes or scales is not 16-byte aligned");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    cudaError_t e = zk::launch_quantize(shard, p->lp, p->quant_format == ZERO_QUANT_FP8_E4M3, p->part, codes, scales,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantize kernel launch");
    return note_work(p, static_cast<cudaStream_t>(stream));
}

zero_status zero_gather_layer_quantized(zero_plan *p, int32_t unit, const int8_t *const *codes,
                                        const float *const *scales, void *out, void *stream) {
    if (!p) return fail(ZERO_EINVAL, "plan is NULL");
    if (p->stage != 3) return fail(ZERO_EINVAL, "the quantized gather needs a stage-3 plan");
    if (p->align % ZERO_QUANT_BLOCK != 0)
        return fail(ZERO_EINVAL, "the quantized gather needs align to be a multiple of %d", ZERO_QUANT_BLOCK);
    if (unit < 0 || unit >= p->n_units()) return fail(ZERO_EINVAL, "unit %d outside [0, %d)", unit, p->n_units());
    const int64_t shard = p->shard_len(unit);
    if (!codes || !scales || (!out && shard > 0)) return fail(ZERO_EINVAL, "NULL codes, scales or output");
    for (int32_t j = 0; j < p->n_ranks; ++j) {
        if (shard > 0 && (!codes[j] || !scales[j])) return fail(ZERO_EINVAL, "codes[%d] or scales[%d] is NULL", j, j);
        if (!aligned16(codes[j]) || !aligned16(scales[j]))
            return fail(ZERO_EALIGN, "codes[%d] or scales[%d] is not 16-byte aligned", j, j);
    }
    if (!aligned16(out)) return fail(ZERO_EALIGN, "out is not 16-byte aligned");
    zero_status st = ensure_device(p);
    if (st != ZERO_OK) return st;
    int64_t off = 0;
    for (int32_t u = 0; u < unit; ++u) off += p->shard_len(u);
    cudaError_t e = zk::launch_dequant_gather(codes, scales, p->n_ranks, p->lp,
                                              p->quant_format == ZERO_QUANT_FP8_E4M3, off, shard, out,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dequantizing gather kernel launch");
    return note_work(p, static_cast<cudaStream_t>(stream));
}

zero_status zero_memory_report(int64_t psi, int32_t n_ranks, int32_t align, double formula_bytes[4],
                               int64_t actual_bytes[4], int64_t comm_elems[4]) {
    if (psi < 0 || n_ranks < 1 || align < 1) return fail(ZERO_EINVAL, "psi < 0, n_ranks < 1 or align < 1");
    const int64_t n = n_ranks;
    // x * psi / n as one rounding: whole part plus the remainder's fraction
    auto per_rank = [&](int64_t mult, int64_t base) {
        const int64_t num = mult * psi;
        return double(base + num / n) + double(num % n) / double(n);
    };
    if (formula_bytes) {
        formula_bytes[0] = double(16 * psi);
        formula_bytes[1] = per_rank(12, 4 * psi);
        formula_bytes[2] = per_rank(14, 2 * psi);
        formula_bytes[3] = per_rank(16, 0);
    }
    if (actual_bytes) {
        const int64_t psi_p = round_up(psi, n * align);
        const int64_t part = psi_p / n;
        actual_bytes[0] = 16 * psi;
        actual_bytes[1] = 4 * psi_p + 12 * part;
        actual_bytes[2] = 2 * psi_p + 14 * part;
        actual_bytes[3] = 16 * part;
    }
    if (comm_elems) {
        comm_elems[0] = 2 * psi;  // all-reduce = reduce-scatter + all-gather
        comm_elems[1] = 2 * psi;
        comm_elems[2] = 2 * psi;
        comm_elems[3] = 3 * psi;  // + one more all-gather (forward and backward)
    }
    return ZERO_OK;
}

void zero_plan_destroy(zero_plan *p) {
    if (!p) return;
    if (p->device >= 0) {
        int cur = 0;
        cudaGetDevice(&cur);
        cudaSetDevice(p->device);
        wait_own_work(p);  // the plan's kernels may still use its scratch
        free_scratch(p);
        for (cudaEvent_t ev : p->spare_events) cudaEventDestroy(ev);
        cudaGetLastError();
        cudaSetDevice(cur);
    }
    delete p;
}

}  // extern "C"
