// Host side of the shard layout: block element counts, the per-parameter
// offset table, ceil-divided equal shards and the packing of a block into
// dp_size zero-padded shards ("vLLM-Omni 发布 Distributed Layerwise Offload…",
// section 2 "weight sharding with AllGather reconstruction"; the cached
// parameter metadata used to re-point views into the rebuilt buffer is from
// section 3).  Plain C++; needs no GPU.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/dlo.h"

namespace dlo {

static thread_local std::string g_last_error;

int set_error(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

}  // namespace dlo

using dlo::set_error;

extern "C" {

const char* dlo_last_error(void) { return dlo::g_last_error.c_str(); }

const char* dlo_status_string(int s) {
    switch (s) {
        case DLO_OK: return "DLO_OK";
        case DLO_ERR_INVALID_ARG: return "DLO_ERR_INVALID_ARG";
        case DLO_ERR_ALIGNMENT: return "DLO_ERR_ALIGNMENT";
        case DLO_ERR_CUDA: return "DLO_ERR_CUDA";
        case DLO_ERR_OOM: return "DLO_ERR_OOM";
        case DLO_ERR_TIMEOUT: return "DLO_ERR_TIMEOUT";
        case DLO_ERR_SHAPE: return "DLO_ERR_SHAPE";
        case DLO_ERR_STATE: return "DLO_ERR_STATE";
        case DLO_ERR_DEVICE_TIMEOUT: return "DLO_ERR_DEVICE_TIMEOUT";
        case DLO_ERR_UNSUPPORTED: return "DLO_ERR_UNSUPPORTED";
        default: return "DLO_ERR_UNKNOWN";
    }
}

int dlo_validate_spec(const dlo_block_spec* s) {
    if (!s) return set_error(DLO_ERR_INVALID_ARG, "spec is null");
    if (s->hidden <= 0 || s->num_heads <= 0 || s->mlp_hidden <= 0 || s->cond_dim <= 0)
        return set_error(DLO_ERR_INVALID_ARG, "spec: every dimension must be positive");
    if (s->hidden % 8 || s->mlp_hidden % 8 || s->cond_dim % 8)
        return set_error(DLO_ERR_ALIGNMENT, "spec: hidden, mlp_hidden and cond_dim must be multiples of 8");
    if (s->hidden % s->num_heads) return set_error(DLO_ERR_SHAPE, "spec: num_heads must divide hidden");
    const int d = s->hidden / s->num_heads;
    if (d != 64 && d != 128) return set_error(DLO_ERR_SHAPE, "spec: head dim %d not 64 or 128", d);
    if (s->cond_dim > 1024) return set_error(DLO_ERR_SHAPE, "spec: cond_dim %d above 1024", s->cond_dim);
    if (s->hidden > 8192) return set_error(DLO_ERR_SHAPE, "spec: hidden %d above 8192", s->hidden);
    if ((int64_t)s->mlp_hidden > (1 << 20)) return set_error(DLO_ERR_SHAPE, "spec: mlp_hidden too large");
    return DLO_OK;
}

int dlo_param_table(const dlo_block_spec* s, int64_t* offsets, int64_t* numels) {
    int st = dlo_validate_spec(s);
    if (st) return st;
    if (!offsets || !numels) return set_error(DLO_ERR_INVALID_ARG, "param_table: null output");
    const int64_t h = s->hidden, m = s->mlp_hidden, C = s->cond_dim;
    const int64_t n[DLO_NUM_PARAMS] = {6 * h * C, 6 * h, 3 * h * h, 3 * h, h * h, h, m * h, m, h * m, h};
    int64_t off = 0;
    for (int i = 0; i < DLO_NUM_PARAMS; ++i) {
        offsets[i] = off;
        numels[i] = n[i];
        off += n[i];
    }
    return DLO_OK;
}

int dlo_block_numel(const dlo_block_spec* s, int64_t* numel) {
    if (!numel) return set_error(DLO_ERR_INVALID_ARG, "block_numel: null output");
    int64_t off[DLO_NUM_PARAMS], n[DLO_NUM_PARAMS];
    int st = dlo_param_table(s, off, n);
    if (st) return st;
    *numel = off[DLO_NUM_PARAMS - 1] + n[DLO_NUM_PARAMS - 1];
    return DLO_OK;
}

int dlo_shard_numel(int64_t numel, int32_t dp_size, int64_t* shard_numel) {
    if (!shard_numel) return set_error(DLO_ERR_INVALID_ARG, "shard_numel: null output");
    if (numel < 0 || dp_size < 1) return set_error(DLO_ERR_INVALID_ARG, "shard_numel: numel >= 0 and dp_size >= 1");
    *shard_numel = numel / dp_size + (numel % dp_size ? 1 : 0);
    return DLO_OK;
}

int dlo_pack_block(const dlo_block_spec* s, const uint16_t* const* params, int32_t dp_size,
                   uint16_t* const* shards) {
    int64_t off[DLO_NUM_PARAMS], n[DLO_NUM_PARAMS];
    int st = dlo_param_table(s, off, n);
    if (st) return st;
    if (!params || !shards) return set_error(DLO_ERR_INVALID_ARG, "pack_block: null pointer array");
    if (dp_size < 1) return set_error(DLO_ERR_INVALID_ARG, "pack_block: dp_size must be >= 1");
    for (int i = 0; i < DLO_NUM_PARAMS; ++i)
        if (!params[i]) return set_error(DLO_ERR_INVALID_ARG, "pack_block: param %d is null", i);
    for (int r = 0; r < dp_size; ++r)
        if (!shards[r]) return set_error(DLO_ERR_INVALID_ARG, "pack_block: shard %d is null", r);
    const int64_t total = off[DLO_NUM_PARAMS - 1] + n[DLO_NUM_PARAMS - 1];
    int64_t S = 0;
    dlo_shard_numel(total, dp_size, &S);
    // Copy every parameter's elements [off, off+n) of the flat buffer into the
    // shards they fall in: flat element f lands in shard f / S at f % S.
    for (int i = 0; i < DLO_NUM_PARAMS; ++i) {
        int64_t f = off[i];
        const int64_t end = off[i] + n[i];
        const uint16_t* src = params[i];
        while (f < end) {
            const int64_t r = f / S;
            const int64_t in_shard = f - r * S;
            int64_t cnt = S - in_shard;
            if (cnt > end - f) cnt = end - f;
            std::memcpy(shards[r] + in_shard, src, (size_t)cnt * sizeof(uint16_t));
            src += cnt;
            f += cnt;
        }
    }
    // Zero padding: everything from flat position `total` to dp*S.
    for (int64_t f = total; f < S * dp_size;) {
        const int64_t r = f / S;
        const int64_t in_shard = f - r * S;
        const int64_t cnt = S - in_shard;
        std::memset(shards[r] + in_shard, 0, (size_t)cnt * sizeof(uint16_t));
        f += cnt;
    }
    return DLO_OK;
}

}  // extern "C"
