"""Thin ctypes binding of ``libmoe_prep.so`` (argument marshalling only).

The functions keep the C names: ``moe_prepare_inputs``, ``moe_batched_experts``,
``moe_topk_reduce``.  Tensors are PyTorch CUDA tensors; only their data
pointers, shapes and strides cross the boundary.  Every step of the path runs
in the library's kernels; if the library is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_prep.so")

MOE_OK = 0
MOE_SF_NONE, MOE_SF_UE8M0_PACKED, MOE_SF_FP32 = 0, 1, 2
MOE_IDS_INT32, MOE_IDS_INT64 = 0, 1
MOE_WEIGHTS_FP32, MOE_WEIGHTS_BF16 = 0, 1
MOE_ACT_SILU = 0
MOE_SHARED_BF16, MOE_SHARED_FP8 = 0, 1
MOE_STAGE_W13, MOE_STAGE_W2, MOE_STAGE_ALL = 1, 2, 3
MOE_DEV_CAPACITY, MOE_DEV_BAD_EXPERT, MOE_DEV_TIMEOUT = 1, 2, 4
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARGUMENT", 2: "MOE_ERR_SHAPE",
                3: "MOE_ERR_UNSUPPORTED", 4: "MOE_ERR_ALIGNMENT", 5: "MOE_ERR_WORKSPACE",
                6: "MOE_ERR_CUDA"}

_i64, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t


class PrepareArgs(ctypes.Structure):
    _fields_ = [
        ("num_tokens", _i64), ("hidden_size", _i64), ("top_k", _i64),
        ("hidden", _vp), ("hidden_stride0", _i64),
        ("topk_ids", _vp), ("topk_ids_dtype", _i32),
        ("topk_ids_stride0", _i64), ("topk_ids_stride1", _i64),
        ("topk_weights", _vp), ("topk_weights_dtype", _i32),
        ("topk_weights_stride0", _i64), ("topk_weights_stride1", _i64),
        ("is_padding", _vp), ("is_padding_stride0", _i64),
        ("x", _vp), ("x_stride0", _i64),
        ("x_sf", _vp), ("sf_mode", _i32), ("x_sf_stride0", _i64), ("x_sf_stride1", _i64),
        ("shared_x_sf", _vp), ("shared_x_sf_stride0", _i64), ("shared_x_sf_stride1", _i64),
        ("shared_x_sf_rows", _i64), ("shared_block_m", _i64),
        ("topk_idx_out", _vp), ("topk_idx_out_stride0", _i64), ("topk_idx_out_stride1", _i64),
        ("topk_weights_out", _vp), ("topk_weights_out_stride0", _i64),
        ("topk_weights_out_stride1", _i64),
        ("logical_to_physical", _vp), ("num_logical", _i64), ("map_stride", _i64),
        ("logical_replica_count", _vp), ("expert_load", _vp), ("num_physical", _i64),
        ("should_record", _vp), ("num_unpadded_tokens", _vp),
        ("num_experts", _i64), ("max_tokens_per_expert", _i64),
        ("x_b", _vp), ("sf_b", _vp), ("expert_num_tokens", _vp), ("route_slot", _vp),
        ("expert_offsets", _vp),
        ("workspace", _vp), ("workspace_bytes", _sz),
        ("device_status", _vp),
    ]


class Nvfp4Args(ctypes.Structure):
    _fields_ = [
        ("num_tokens", _i64), ("hidden_size", _i64), ("top_k", _i64),
        ("hidden", _vp), ("hidden_stride0", _i64),
        ("topk_ids", _vp), ("topk_ids_dtype", _i32),
        ("topk_ids_stride0", _i64), ("topk_ids_stride1", _i64),
        ("topk_weights", _vp), ("topk_weights_dtype", _i32),
        ("topk_weights_stride0", _i64), ("topk_weights_stride1", _i64),
        ("is_padding", _vp), ("is_padding_stride0", _i64),
        ("x", _vp), ("x_stride0", _i64),
        ("x_sf", _vp), ("x_sf_stride0", _i64),
        ("x_scales", _vp),
        ("shared_x", _vp), ("shared_x_stride0", _i64), ("shared_x_dtype", _i32),
        ("shared_x_sf", _vp), ("shared_x_sf_stride0", _i64), ("shared_x_sf_stride1", _i64),
        ("shared_x_sf_rows", _i64), ("shared_block_m", _i64),
        ("topk_idx_out", _vp), ("topk_idx_out_stride0", _i64), ("topk_idx_out_stride1", _i64),
        ("topk_weights_out", _vp), ("topk_weights_out_stride0", _i64),
        ("topk_weights_out_stride1", _i64),
        ("logical_to_physical", _vp), ("num_logical", _i64), ("map_stride", _i64),
        ("logical_replica_count", _vp), ("expert_load", _vp), ("num_physical", _i64),
        ("should_record", _vp), ("num_unpadded_tokens", _vp),
        ("w2_global_scale", _vp), ("l2_alpha", _vp), ("num_local_experts", _i64),
        ("l2_activation_scale", ctypes.c_float),
        ("device_status", _vp),
    ]


class ExpertsArgs(ctypes.Structure):
    _fields_ = [
        ("num_experts", _i64), ("max_tokens_per_expert", _i64), ("hidden_size", _i64),
        ("intermediate_size", _i64), ("activation", _i32), ("stages", _i32),
        ("output", _vp), ("hidden", _vp), ("a_scale", _vp), ("a_scale_mode", _i32),
        ("w13", _vp), ("w13_scale", _vp), ("w2", _vp), ("w2_scale", _vp),
        ("expert_num_tokens", _vp), ("expert_offsets", _vp),
        ("inter_q", _vp), ("inter_sf", _vp),
        ("workspace13", _vp), ("workspace13_bytes", _sz),
        ("workspace2", _vp), ("workspace2_bytes", _sz),
        ("valid_shape_m", _i64), ("gate_up_dump", _vp), ("device_status", _vp),
    ]


_lib = None


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    _lib = configure(ctypes.CDLL(LIB_PATH))
    return _lib


def configure(lib):
    """Declare the C signatures on a loaded copy of the library."""
    lib.moe_abi_version.restype = ctypes.c_int
    lib.moe_last_error.restype = ctypes.c_char_p
    lib.moe_prepare_inputs.restype = ctypes.c_int
    lib.moe_prepare_inputs.argtypes = [ctypes.POINTER(PrepareArgs), _vp]
    lib.moe_prepare_workspace_size.restype = _sz
    lib.moe_prepare_workspace_size.argtypes = [_i64, _i64, _i64]
    lib.moe_prepare_inputs_noalloc.restype = ctypes.c_int
    lib.moe_prepare_inputs_noalloc.argtypes = [ctypes.POINTER(PrepareArgs), _vp]
    lib.moe_batched_experts.restype = ctypes.c_int
    lib.moe_batched_experts.argtypes = [ctypes.POINTER(ExpertsArgs), _vp]
    lib.moe_batched_experts_workspace_size.restype = _sz
    lib.moe_batched_experts_workspace_size.argtypes = [_i64, _i64, _i64, _i64, _i64,
                                                       ctypes.c_int]
    lib.moe_topk_reduce.restype = ctypes.c_int
    lib.moe_topk_reduce.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _i64, _i64, _vp, _vp,
                                    _vp]
    return lib


class MoeError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(fn, st):
    if st != MOE_OK:
        raise MoeError(fn, st, load().moe_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def prepare_workspace_size(num_tokens, top_k, num_experts) -> int:
    return int(load().moe_prepare_workspace_size(num_tokens, top_k, num_experts))


def experts_workspace_size(E, M_max, K, N, valid_shape_m, which) -> int:
    return int(load().moe_batched_experts_workspace_size(E, M_max, K, N, valid_shape_m, which))


def moe_prepare_inputs(hidden, topk_ids, topk_weights, x, x_sf, topk_idx_out, topk_weights_out,
                       is_padding=None, sf_mode=MOE_SF_UE8M0_PACKED, eplb=None, dispatch=None,
                       device_status=None, stream=None, shared_x_sf=None, shared_block_m=None):
    """Input staging (and optional dispatch).  See include/moe_prep.h.

    shared_x_sf: uint8 [rows, K/128] shared-expert scale pages, given together
    with shared_block_m (UE8M0 scales only).

    eplb: dict(logical_to_physical, logical_replica_count, expert_load=None,
               should_record=None, num_unpadded_tokens=None) -- device tensors.
    dispatch: dict(num_experts, max_tokens_per_expert, x_b, sf_b, expert_num_tokens,
                   route_slot, workspace[, expert_offsets]) -- with expert_offsets
              ([E+1] int32) the rows are laid out contiguously per expert.
    """
    T, K = hidden.shape
    a = PrepareArgs()
    a.num_tokens, a.hidden_size = T, K
    a.top_k = topk_ids.shape[1] if topk_ids.dim() == 2 else 0
    a.hidden, a.hidden_stride0 = _ptr(hidden), hidden.stride(0)
    a.topk_ids = _ptr(topk_ids)
    a.topk_ids_dtype = MOE_IDS_INT64 if topk_ids.dtype == torch.int64 else MOE_IDS_INT32
    a.topk_ids_stride0, a.topk_ids_stride1 = topk_ids.stride(0), topk_ids.stride(1)
    a.topk_weights = _ptr(topk_weights)
    a.topk_weights_dtype = MOE_WEIGHTS_BF16 if topk_weights.dtype == torch.bfloat16 else \
        MOE_WEIGHTS_FP32
    a.topk_weights_stride0, a.topk_weights_stride1 = topk_weights.stride(0), topk_weights.stride(1)
    if is_padding is not None:
        a.is_padding, a.is_padding_stride0 = _ptr(is_padding), is_padding.stride(0)
    a.x, a.x_stride0 = _ptr(x), x.stride(0)
    a.sf_mode = sf_mode
    if x_sf is not None:
        a.x_sf, a.x_sf_stride0 = _ptr(x_sf), x_sf.stride(0)
        a.x_sf_stride1 = x_sf.stride(1) if x_sf.dim() > 1 else 1
    a.topk_idx_out = _ptr(topk_idx_out)
    a.topk_idx_out_stride0, a.topk_idx_out_stride1 = topk_idx_out.stride(0), topk_idx_out.stride(1)
    a.topk_weights_out = _ptr(topk_weights_out)
    a.topk_weights_out_stride0 = topk_weights_out.stride(0)
    a.topk_weights_out_stride1 = topk_weights_out.stride(1)
    if shared_x_sf is not None:
        a.shared_x_sf = _ptr(shared_x_sf)
        a.shared_x_sf_stride0, a.shared_x_sf_stride1 = shared_x_sf.stride(0), shared_x_sf.stride(1)
        a.shared_x_sf_rows = shared_x_sf.shape[0]
    if shared_block_m is not None:
        a.shared_block_m = int(shared_block_m)
    if eplb:
        l2p = eplb["logical_to_physical"]
        a.logical_to_physical, a.num_logical, a.map_stride = _ptr(l2p), l2p.shape[0], l2p.stride(0)
        a.logical_replica_count = _ptr(eplb["logical_replica_count"])
        load_t = eplb.get("expert_load")
        if load_t is not None:
            a.expert_load, a.num_physical = _ptr(load_t), load_t.numel()
        a.should_record = _ptr(eplb.get("should_record"))
        a.num_unpadded_tokens = _ptr(eplb.get("num_unpadded_tokens"))
    if dispatch:
        a.num_experts = dispatch["num_experts"]
        a.max_tokens_per_expert = dispatch["max_tokens_per_expert"]
        a.x_b, a.sf_b = _ptr(dispatch["x_b"]), _ptr(dispatch["sf_b"])
        a.expert_num_tokens = _ptr(dispatch["expert_num_tokens"])
        a.route_slot = _ptr(dispatch["route_slot"])
        a.expert_offsets = _ptr(dispatch.get("expert_offsets"))
        ws = dispatch["workspace"]
        a.workspace, a.workspace_bytes = _ptr(ws), ws.numel() * ws.element_size()
    a.device_status = _ptr(device_status)
    _check("moe_prepare_inputs", load().moe_prepare_inputs(ctypes.byref(a), _stream(stream)))


def moe_prepare_inputs_noalloc(hidden, topk_ids, topk_weights, x, x_sf, topk_idx_out,
                               topk_weights_out, is_padding=None, sf_mode=MOE_SF_UE8M0_PACKED,
                               eplb=None, dispatch=None, device_status=None, stream=None):
    """Staging + dispatch for callers that cannot allocate device memory.

    Same arguments as ``moe_prepare_inputs`` except that ``dispatch`` needs no
    ``workspace``: the scratch of the dispatch is a fixed array inside the
    library (MOE_PREPARE_NOALLOC_SCRATCH_BYTES, 4 MiB, per GPU).  Calls on one
    device share that array, so calls that may overlap on the GPU must be
    serialised; the first call on a device looks the array up, so make it
    before any stream capture.
    """
    T, K = hidden.shape
    a = PrepareArgs()
    a.num_tokens, a.hidden_size = T, K
    a.top_k = topk_ids.shape[1] if topk_ids.dim() == 2 else 0
    a.hidden, a.hidden_stride0 = _ptr(hidden), hidden.stride(0)
    a.topk_ids = _ptr(topk_ids)
    a.topk_ids_dtype = MOE_IDS_INT64 if topk_ids.dtype == torch.int64 else MOE_IDS_INT32
    a.topk_ids_stride0, a.topk_ids_stride1 = topk_ids.stride(0), topk_ids.stride(1)
    a.topk_weights = _ptr(topk_weights)
    a.topk_weights_dtype = MOE_WEIGHTS_BF16 if topk_weights.dtype == torch.bfloat16 else \
        MOE_WEIGHTS_FP32
    a.topk_weights_stride0, a.topk_weights_stride1 = topk_weights.stride(0), topk_weights.stride(1)
    if is_padding is not None:
        a.is_padding, a.is_padding_stride0 = _ptr(is_padding), is_padding.stride(0)
    a.x, a.x_stride0 = _ptr(x), x.stride(0)
    a.sf_mode = sf_mode
    if x_sf is not None:
        a.x_sf, a.x_sf_stride0 = _ptr(x_sf), x_sf.stride(0)
        a.x_sf_stride1 = x_sf.stride(1) if x_sf.dim() > 1 else 1
    a.topk_idx_out = _ptr(topk_idx_out)
    a.topk_idx_out_stride0, a.topk_idx_out_stride1 = topk_idx_out.stride(0), topk_idx_out.stride(1)
    a.topk_weights_out = _ptr(topk_weights_out)
    a.topk_weights_out_stride0 = topk_weights_out.stride(0)
    a.topk_weights_out_stride1 = topk_weights_out.stride(1)
    if eplb:
        l2p = eplb["logical_to_physical"]
        a.logical_to_physical, a.num_logical, a.map_stride = _ptr(l2p), l2p.shape[0], l2p.stride(0)
        a.logical_replica_count = _ptr(eplb["logical_replica_count"])
        load_t = eplb.get("expert_load")
        if load_t is not None:
            a.expert_load, a.num_physical = _ptr(load_t), load_t.numel()
        a.should_record = _ptr(eplb.get("should_record"))
        a.num_unpadded_tokens = _ptr(eplb.get("num_unpadded_tokens"))
    if dispatch:
        a.num_experts = dispatch["num_experts"]
        a.max_tokens_per_expert = dispatch["max_tokens_per_expert"]
        a.x_b, a.sf_b = _ptr(dispatch["x_b"]), _ptr(dispatch["sf_b"])
        a.expert_num_tokens = _ptr(dispatch["expert_num_tokens"])
        a.route_slot = _ptr(dispatch["route_slot"])
    a.device_status = _ptr(device_status)
    _check("moe_prepare_inputs_noalloc",
           load().moe_prepare_inputs_noalloc(ctypes.byref(a), _stream(stream)))


def moe_prepare_nvfp4_inputs(hidden, topk_ids, topk_weights, x, x_sf, x_scales, topk_idx_out,
                             topk_weights_out, is_padding=None, shared_x=None, eplb=None,
                             w2_global_scale=None, l2_alpha=None, l2_activation_scale=1.0,
                             device_status=None, stream=None, shared_x_sf=None,
                             shared_block_m=None):
    """NVFP4 token staging (E2M1 + E4M3 per 16 + fp32 per-token scale) and the
    top-k repack.  x: uint8 [T, K/2]; x_sf: int32 [T, K/64]; x_scales: fp32 [T].
    shared_x: bf16 [T, K] (a copy of the hidden rows) or uint8 [T, K] (the
    MXFP8 shared input, fp8 codes, given with shared_x_sf uint8 [rows, K/128]
    and shared_block_m).  See include/moe_prep.h."""
    T, K = hidden.shape
    a = Nvfp4Args()
    a.num_tokens, a.hidden_size = T, K
    a.top_k = topk_ids.shape[1] if topk_ids.dim() == 2 else 0
    a.hidden, a.hidden_stride0 = _ptr(hidden), hidden.stride(0)
    a.topk_ids = _ptr(topk_ids)
    a.topk_ids_dtype = MOE_IDS_INT64 if topk_ids.dtype == torch.int64 else MOE_IDS_INT32
    a.topk_ids_stride0, a.topk_ids_stride1 = topk_ids.stride(0), topk_ids.stride(1)
    a.topk_weights = _ptr(topk_weights)
    a.topk_weights_dtype = MOE_WEIGHTS_BF16 if topk_weights.dtype == torch.bfloat16 else \
        MOE_WEIGHTS_FP32
    a.topk_weights_stride0, a.topk_weights_stride1 = topk_weights.stride(0), topk_weights.stride(1)
    if is_padding is not None:
        a.is_padding, a.is_padding_stride0 = _ptr(is_padding), is_padding.stride(0)
    a.x, a.x_stride0 = _ptr(x), x.stride(0)
    a.x_sf, a.x_sf_stride0 = _ptr(x_sf), x_sf.stride(0)
    a.x_scales = _ptr(x_scales)
    if shared_x is not None:
        a.shared_x, a.shared_x_stride0 = _ptr(shared_x), shared_x.stride(0)
        a.shared_x_dtype = MOE_SHARED_BF16 if shared_x.dtype == torch.bfloat16 else MOE_SHARED_FP8
    if shared_x_sf is not None:
        a.shared_x_sf = _ptr(shared_x_sf)
        a.shared_x_sf_stride0, a.shared_x_sf_stride1 = shared_x_sf.stride(0), shared_x_sf.stride(1)
        a.shared_x_sf_rows = shared_x_sf.shape[0]
    if shared_block_m is not None:
        a.shared_block_m = int(shared_block_m)
    a.topk_idx_out = _ptr(topk_idx_out)
    a.topk_idx_out_stride0, a.topk_idx_out_stride1 = topk_idx_out.stride(0), topk_idx_out.stride(1)
    a.topk_weights_out = _ptr(topk_weights_out)
    a.topk_weights_out_stride0 = topk_weights_out.stride(0)
    a.topk_weights_out_stride1 = topk_weights_out.stride(1)
    if eplb:
        l2p = eplb["logical_to_physical"]
        a.logical_to_physical, a.num_logical, a.map_stride = _ptr(l2p), l2p.shape[0], l2p.stride(0)
        a.logical_replica_count = _ptr(eplb["logical_replica_count"])
        load_t = eplb.get("expert_load")
        if load_t is not None:
            a.expert_load, a.num_physical = _ptr(load_t), load_t.numel()
        a.should_record = _ptr(eplb.get("should_record"))
        a.num_unpadded_tokens = _ptr(eplb.get("num_unpadded_tokens"))
    if l2_alpha is not None:
        a.w2_global_scale, a.l2_alpha = _ptr(w2_global_scale), _ptr(l2_alpha)
        a.num_local_experts = l2_alpha.numel()
    a.l2_activation_scale = float(l2_activation_scale)
    a.device_status = _ptr(device_status)
    _check("moe_prepare_nvfp4_inputs",
           load().moe_prepare_nvfp4_inputs(ctypes.byref(a), _stream(stream)))


def moe_batched_experts(output, hidden, a_scale, w13, w13_scale, w2, w2_scale,
                        expert_num_tokens, workspace13=None, workspace2=None, valid_shape_m=0,
                        inter_q=None, inter_sf=None, gate_up_dump=None, stages=MOE_STAGE_ALL,
                        device_status=None, stream=None, expert_offsets=None):
    """w13 GEMM + SiLU-and-mul requant + w2 GEMM.  See include/moe_prep.h.

    expert_offsets ([E+1] int32, nullable) selects the contiguous layout.
    """
    E = w13.shape[0]
    K = w13.shape[2]
    N = w2.shape[2]
    if output is not None:
        M_max = output.shape[1] if output.dim() == 3 else output.shape[0] // E
    else:
        M_max = hidden.shape[0] // E
    a = ExpertsArgs()
    a.num_experts, a.max_tokens_per_expert, a.hidden_size, a.intermediate_size = E, M_max, K, N
    a.activation, a.stages = MOE_ACT_SILU, stages
    a.output, a.hidden, a.a_scale = _ptr(output), _ptr(hidden), _ptr(a_scale)
    # fp32 activation scales [E*M_max, K/128] select the fp32 dequantisation
    a.a_scale_mode = (MOE_SF_FP32 if a_scale is not None and a_scale.dtype == torch.float32
                      else MOE_SF_UE8M0_PACKED)
    a.w13, a.w13_scale, a.w2, a.w2_scale = _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale)
    a.expert_num_tokens = _ptr(expert_num_tokens)
    a.expert_offsets = _ptr(expert_offsets)
    a.inter_q, a.inter_sf = _ptr(inter_q), _ptr(inter_sf)
    if workspace13 is not None:
        a.workspace13 = _ptr(workspace13)
        a.workspace13_bytes = workspace13.numel() * workspace13.element_size()
    if workspace2 is not None:
        a.workspace2 = _ptr(workspace2)
        a.workspace2_bytes = workspace2.numel() * workspace2.element_size()
    a.valid_shape_m = valid_shape_m
    a.gate_up_dump = _ptr(gate_up_dump)
    a.device_status = _ptr(device_status)
    _check("moe_batched_experts", load().moe_batched_experts(ctypes.byref(a), _stream(stream)))


def moe_topk_reduce(expert_out, topk_idx, route_slot, topk_weights, out, stream=None,
                    num_valid_tokens=None):
    """Top-k weighted sum back to token order.  See include/moe_prep.h.

    topk_idx None: route_slot holds rows of expert_out (contiguous layout).
    num_valid_tokens: optional int32 device scalar; tokens at or past it are
    not written.
    """
    if expert_out.dim() == 3:
        E, M_max, K = expert_out.shape
    else:
        (E, K), M_max = (1, expert_out.shape[1]), expert_out.shape[0]
    T, k = route_slot.shape
    _check("moe_topk_reduce", load().moe_topk_reduce(
        _ptr(expert_out), E, M_max, K, _ptr(topk_idx), _ptr(route_slot), _ptr(topk_weights), T, k,
        _ptr(num_valid_tokens), _ptr(out), _stream(stream)))


class MoeLayer:
    """Device buffers of one batched MoE expert layer and the three calls.

    ``forward`` runs staging + dispatch, the batched experts and the top-k
    reduce on the current stream and returns the bf16 [T, K] output.
    """

    def __init__(self, T, K, N, E, top_k, M_max, w13, w13_s, w2, w2_s, device="cuda",
                 valid_shape_m=None, eplb=None, contiguous=False, fp32_scales=False):
        # contiguous: rows are packed per expert (expert_offsets); the buffers
        # hold E * ceil(T*k/E) rows, whatever the per-expert load
        if contiguous:
            M_max = max(1, -(-(T * top_k) // E))
        self.contiguous = contiguous
        # fp32_scales: 1x128 activation scales kept as fp32 (amax / 448) instead
        # of packed UE8M0 exponents
        self.sf_mode = MOE_SF_FP32 if fp32_scales else MOE_SF_UE8M0_PACKED
        self.T, self.K, self.N, self.E, self.top_k, self.M_max = T, K, N, E, top_k, M_max
        self.w13, self.w13_s, self.w2, self.w2_s = w13, w13_s, w2, w2_s
        self.eplb = eplb
        G = K // 128
        W = (G + 3) // 4
        dev = torch.device(device)
        u8 = dict(dtype=torch.uint8, device=dev)
        self.x = torch.empty((T, K), **u8)
        self.x_sf = (torch.empty((T, G), dtype=torch.float32, device=dev) if fp32_scales else
                     torch.empty((T, W), dtype=torch.int32, device=dev))
        self.ids_out = torch.empty((T, top_k), dtype=torch.int64, device=dev)
        self.w_out = torch.empty((T, top_k), dtype=torch.float32, device=dev)
        self.x_b = torch.empty((E * M_max, K), **u8)
        self.sf_b = (torch.empty((E * M_max, G), dtype=torch.float32, device=dev) if fp32_scales
                     else torch.empty((E * M_max, W), dtype=torch.int32, device=dev))
        self.expert_num_tokens = torch.zeros(E, dtype=torch.int32, device=dev)
        self.route_slot = torch.empty((T, top_k), dtype=torch.int32, device=dev)
        self.expert_offsets = (torch.zeros(E + 1, dtype=torch.int32, device=dev) if contiguous
                               else None)
        self.ws_prep = torch.empty(max(prepare_workspace_size(T, top_k, E), 256), **u8)
        self.valid_shape_m = valid_shape_m if valid_shape_m is not None else T * top_k
        self.ws13 = torch.empty(experts_workspace_size(E, M_max, K, N, self.valid_shape_m, 13), **u8)
        self.ws2 = torch.zeros(max(experts_workspace_size(E, M_max, K, N, self.valid_shape_m, 2),
                                   256), **u8)
        self.out_b = torch.empty((E, M_max, K), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def dispatch_args(self):
        return dict(num_experts=self.E, max_tokens_per_expert=self.M_max, x_b=self.x_b,
                    sf_b=self.sf_b, expert_num_tokens=self.expert_num_tokens,
                    route_slot=self.route_slot, workspace=self.ws_prep,
                    expert_offsets=self.expert_offsets)

    def prepare(self, hidden, topk_ids, topk_weights, is_padding=None, stream=None):
        moe_prepare_inputs(hidden, topk_ids, topk_weights, self.x, self.x_sf, self.ids_out,
                           self.w_out, is_padding=is_padding, sf_mode=self.sf_mode,
                           eplb=self.eplb, dispatch=self.dispatch_args(),
                           device_status=self.status, stream=stream)

    def experts(self, gate_up_dump=None, stream=None):
        moe_batched_experts(self.out_b, self.x_b, self.sf_b, self.w13, self.w13_s, self.w2,
                            self.w2_s, self.expert_num_tokens, self.ws13, self.ws2,
                            valid_shape_m=self.valid_shape_m, gate_up_dump=gate_up_dump,
                            device_status=self.status, stream=stream,
                            expert_offsets=self.expert_offsets)

    def reduce(self, stream=None):
        moe_topk_reduce(self.out_b, None if self.contiguous else self.ids_out, self.route_slot,
                        self.w_out, self.out, stream=stream)

    def forward(self, hidden, topk_ids, topk_weights, is_padding=None, stream=None):
        self.prepare(hidden, topk_ids, topk_weights, is_padding, stream)
        self.experts(stream=stream)
        self.reduce(stream=stream)
        return self.out

    def inter(self):
        """(inter_q, inter_sf) views of workspace13 as written by the w13 stage."""
        EM, N = self.E * self.M_max, self.N
        off = ((EM * N + 255) // 256) * 256
        Wy = (N // 128 + 3) // 4
        q = self.ws13[:EM * N].view(EM, N)
        sf = self.ws13[off:off + EM * Wy * 4].view(torch.int32).view(EM, Wy)
        return q, sf

    def forward_host(self, hidden_h, topk_ids_h, topk_weights_h, is_padding_h, out_h,
                     stream=None, chunks=None):
        """End-to-end call from pinned host buffers: copy the step's inputs to
        the device, run the three stages, copy the bf16 output back into
        ``out_h`` (pinned).  Nothing synchronises with the host.

        The reduce runs in token chunks (``chunks``; by default 4 from 1024
        tokens on, else 1), and each chunk's output rows go back to the host
        on a second stream while the next chunk is reduced (prefill: the
        output copy then costs 0.13 ms less).  The call's stream waits for the
        last copy, so work queued on it afterwards, or a synchronisation of
        it, sees ``out_h`` complete."""
        s = stream if stream is not None else torch.cuda.current_stream()
        if not hasattr(self, "_in_dev"):
            dev = self.x.device
            self._in_dev = (torch.empty(hidden_h.shape, dtype=hidden_h.dtype, device=dev),
                            torch.empty(topk_ids_h.shape, dtype=topk_ids_h.dtype, device=dev),
                            torch.empty(topk_weights_h.shape, dtype=topk_weights_h.dtype,
                                        device=dev),
                            None if is_padding_h is None else
                            torch.empty(is_padding_h.shape, dtype=is_padding_h.dtype, device=dev))
            self._copy_stream = torch.cuda.Stream(device=dev)
        h, i, w, p = self._in_dev
        with torch.cuda.stream(s):
            h.copy_(hidden_h, non_blocking=True)
            i.copy_(topk_ids_h, non_blocking=True)
            w.copy_(topk_weights_h, non_blocking=True)
            if p is not None:
                p.copy_(is_padding_h, non_blocking=True)
        self.prepare(h, i, w, p, stream=s)
        self.experts(stream=s)
        T = self.out.shape[0]
        n = chunks if chunks is not None else (4 if T >= 1024 else 1)
        n = max(1, min(n, T))
        if n == 1:
            self.reduce(stream=s)
            with torch.cuda.stream(s):
                out_h.copy_(self.out, non_blocking=True)
            return out_h
        cs = self._copy_stream
        idx = None if self.contiguous else self.ids_out
        bounds = [T * c // n for c in range(n + 1)]
        for c in range(n):
            t0, t1 = bounds[c], bounds[c + 1]
            moe_topk_reduce(self.out_b, None if idx is None else idx[t0:t1],
                            self.route_slot[t0:t1], self.w_out[t0:t1], self.out[t0:t1],
                            stream=s)
            cs.wait_stream(s)
            with torch.cuda.stream(cs):
                out_h[t0:t1].copy_(self.out[t0:t1], non_blocking=True)
        s.wait_stream(cs)
        return out_h
