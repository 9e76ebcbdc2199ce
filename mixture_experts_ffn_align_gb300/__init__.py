"""Python binding of the GB300 fused MoE expert forward (libmoe_ffn.so).

Argument marshalling only: every function here has the name of a C entry
point in ``include/moe_ffn.h``, takes torch tensors (device memory) or None,
passes their data pointers and the current CUDA stream to the library, and
raises ``MoEError`` on a non-OK status.  All computation happens in the CUDA
kernels of the library; there is no fallback.  The library must have been
built (``__graft_entry__.build()`` or ``python -m
mixture_experts_ffn_align_gb300._build``); importing a function that needs it
raises if it is missing.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_ffn.so")

QUANT = {"bf16": 0, "fp8": 1, "mxfp4": 2, "mxfp8": 3}
SCALE_FMT = {"fp32": 0, "ue8m0": 1}

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_DEVICE_TIMEOUT", 5: "MOE_ERR_WORKSPACE_TOO_SMALL",
          6: "MOE_ERR_DEVICE_BAD_INDEX"}

EXPORTS = ["moe_m_sum_bound", "moe_align_workspace_bytes", "moe_align_permute_launches",
           "moe_workspace_bytes",
           "moe_host_workspace_bytes", "moe_align_permute", "grouped_gemm_w13", "act_mul_quant",
           "grouped_gemm_w2", "unpermute_reduce", "fused_experts", "fused_experts_from_host",
           "moe_sync_status", "moe_status_string", "moe_debug_set_watchdog",
           "moe_debug_set_bf16_gemm_form",
           "moe_align_permute_noalloc", "moe_last_error_string", "moe_topk_router",
           "moe_batched_workspace_bytes", "fused_experts_batched", "grouped_gemm_w13_ex",
           "grouped_gemm_w2_ex", "fused_experts_ex", "moe_gemm2_splits",
           "moe_gemm2_partial_bytes", "grouped_gemm_w2_split", "unpermute_reduce_split",
           "moe_prepacked_scale_bytes", "moe_prepack_weights"]

NOALLOC_SCRATCH_BYTES = 1 << 20   # MOE_NOALLOC_SCRATCH_BYTES in include/moe_ffn.h


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))


class CProblem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("M", "H", "I", "E", "topk", "block_size", "quant", "act_scale_fmt",
                 "apply_router_weight_on_input", "router_weight_in_gemm2", "act_recipe")] + \
               [(n, ctypes.c_float) for n in ("gemm1_alpha", "gemm1_beta", "gemm1_clamp_limit")] + \
               [("weight_scales_prepacked", ctypes.c_int32)]


@dataclass(frozen=True)
class Problem:
    """Mirror of ``moe_problem``."""
    M: int
    H: int
    I: int
    E: int
    topk: int
    block_size: int = 128
    quant: str = "bf16"
    act_scale_fmt: str = "fp32"
    apply_router_weight_on_input: bool = False
    router_weight_in_gemm2: bool = False
    # None: SiLU(gate) * up; else (alpha, beta, clamp_limit) of the gemm1 recipe
    act_recipe: tuple | None = None
    # MXFP4 / MXFP8: the weight scales passed are moe_prepack_weights' output
    weight_scales_prepacked: bool = False

    def c(self) -> CProblem:
        a, b, lim = self.act_recipe if self.act_recipe is not None else (0.0, 0.0, 0.0)
        return CProblem(self.M, self.H, self.I, self.E, self.topk, self.block_size,
                        QUANT[self.quant], SCALE_FMT[self.act_scale_fmt],
                        int(self.apply_router_weight_on_input),
                        int(self.router_weight_in_gemm2), int(self.act_recipe is not None),
                        float(a), float(b), float(lim), int(self.weight_scales_prepacked))

    @classmethod
    def from_config(cls, cfg, **kw):
        d = dict(M=cfg.M, H=cfg.H, I=cfg.I, E=cfg.E, topk=cfg.topk, block_size=cfg.block_size,
                 quant=cfg.quant, act_scale_fmt=cfg.act_scale_fmt,
                 apply_router_weight_on_input=cfg.apply_router_weight_on_input)
        d.update(kw)
        return cls(**d)


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe_ffn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(CProblem)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        for n in ("moe_m_sum_bound", "moe_align_workspace_bytes", "moe_workspace_bytes",
                  "moe_host_workspace_bytes"):
            getattr(L, n).argtypes, getattr(L, n).restype = [P], sz
        L.moe_align_permute.argtypes = [P] + [vp] * 10 + [vp, sz, vp]
        L.moe_align_permute_noalloc.argtypes = [P] + [vp] * 10 + [vp]
        L.moe_align_permute_noalloc.restype = i32
        L.grouped_gemm_w13.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp]
        L.act_mul_quant.argtypes = [P, vp, vp, vp, vp, vp]
        L.grouped_gemm_w2.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
        L.unpermute_reduce.argtypes = [P, vp, vp, vp, vp, vp]
        L.fused_experts.argtypes = [P] + [vp] * 9 + [sz, vp]
        L.fused_experts_from_host.argtypes = [P] + [vp] * 9 + [sz, vp]
        L.moe_sync_status.argtypes = [vp]
        L.moe_prepacked_scale_bytes.argtypes = [P, i32]
        L.moe_prepacked_scale_bytes.restype = sz
        L.moe_prepack_weights.argtypes = [P, vp, vp, vp, vp, vp]
        L.moe_topk_router.argtypes = [i32, i32, i32, vp, i32, i32, i32, vp, vp, vp, vp, vp]
        L.moe_batched_workspace_bytes.argtypes = [P, i32]
        L.moe_batched_workspace_bytes.restype = sz
        L.fused_experts_batched.argtypes = [P, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.grouped_gemm_w13_ex.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp]
        L.grouped_gemm_w2_ex.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.fused_experts_ex.argtypes = [P] + [vp] * 11 + [sz, vp]
        L.moe_gemm2_splits.argtypes, L.moe_gemm2_splits.restype = [P], i32
        L.moe_align_permute_launches.argtypes = [P]
        L.moe_align_permute_launches.restype = i32
        L.moe_gemm2_partial_bytes.argtypes, L.moe_gemm2_partial_bytes.restype = [P, i32], sz
        L.grouped_gemm_w2_split.argtypes = [P, vp, vp, vp, vp, vp, i32, vp, vp]
        L.unpermute_reduce_split.argtypes = [P, vp, i32, vp, vp, vp, vp]
        L.moe_status_string.argtypes, L.moe_status_string.restype = [i32], ctypes.c_char_p
        L.moe_last_error_string.argtypes, L.moe_last_error_string.restype = [], ctypes.c_char_p
        L.moe_debug_set_watchdog.argtypes, L.moe_debug_set_watchdog.restype = \
            [ctypes.c_int64, i32], None
        L.moe_debug_set_bf16_gemm_form.argtypes, L.moe_debug_set_bf16_gemm_form.restype = \
            [i32], None
        for n in ("moe_align_permute", "grouped_gemm_w13", "act_mul_quant", "grouped_gemm_w2",
                  "unpermute_reduce", "fused_experts", "fused_experts_from_host",
                  "moe_sync_status", "moe_topk_router", "fused_experts_batched",
                  "grouped_gemm_w13_ex", "grouped_gemm_w2_ex", "fused_experts_ex",
                  "grouped_gemm_w2_split", "unpermute_reduce_split", "moe_prepack_weights"):
            getattr(L, n).restype = i32
        _lib = L
    return _lib


def _p(t):
    """Data pointer of a tensor (or None -> NULL)."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        detail = moe_last_error_string() if status == 3 else ""
        raise MoEError(status, where, detail)


def _cp(p: Problem):
    return ctypes.byref(p.c())


# ------------------------------------------------------------------ sizes
def moe_m_sum_bound(p: Problem) -> int:
    return int(lib().moe_m_sum_bound(_cp(p)))


def moe_align_workspace_bytes(p: Problem) -> int:
    return int(lib().moe_align_workspace_bytes(_cp(p)))


def moe_align_permute_launches(p: Problem) -> int:
    """Kernels moe_align_permute launches for p (routing + permute)."""
    return int(lib().moe_align_permute_launches(_cp(p)))


def moe_workspace_bytes(p: Problem) -> int:
    return int(lib().moe_workspace_bytes(_cp(p)))


def moe_host_workspace_bytes(p: Problem) -> int:
    return int(lib().moe_host_workspace_bytes(_cp(p)))


def moe_prepacked_scale_bytes(p: Problem, which: int) -> int:
    """Bytes of the prepacked w13 (which=0) or w2 (which=1) weight scales."""
    return int(lib().moe_prepacked_scale_bytes(_cp(p), int(which)))


def moe_prepack_weights(p: Problem, w13_scale, w2_scale, w13_scale_packed, w2_scale_packed,
                        stream=None):
    _check(lib().moe_prepack_weights(_cp(p), _p(w13_scale), _p(w2_scale), _p(w13_scale_packed),
                                     _p(w2_scale_packed), _stream(stream)),
           "moe_prepack_weights")


# ------------------------------------------------------------------ stages
def moe_align_permute(p: Problem, x, topk_ids, topk_weights, sorted_ids, block_expert_ids,
                      expert_offsets, num_post_padded, inv_perm, x_perm, x_perm_scale,
                      workspace, stream=None):
    _check(lib().moe_align_permute(
        _cp(p), _p(x), _p(topk_ids), _p(topk_weights), _p(sorted_ids), _p(block_expert_ids),
        _p(expert_offsets), _p(num_post_padded), _p(inv_perm), _p(x_perm), _p(x_perm_scale),
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "moe_align_permute")


def moe_align_permute_noalloc(p: Problem, x, topk_ids, topk_weights, sorted_ids,
                              block_expert_ids, expert_offsets, num_post_padded, inv_perm,
                              x_perm, x_perm_scale, stream=None):
    """moe_align_permute without a workspace, for callers that may not
    allocate device memory at call time (for instance an engine that owns the
    whole device through its own memory pool).  Its scratch is a fixed
    MOE_NOALLOC_SCRATCH_BYTES array inside the library, shared by every call on
    a device; larger problems raise MoEError(MOE_ERR_WORKSPACE_TOO_SMALL).
    Make the first call on a device before any stream capture, and keep calls
    ordered on one stream (overlapping calls race on the shared array)."""
    _check(lib().moe_align_permute_noalloc(
        _cp(p), _p(x), _p(topk_ids), _p(topk_weights), _p(sorted_ids), _p(block_expert_ids),
        _p(expert_offsets), _p(num_post_padded), _p(inv_perm), _p(x_perm), _p(x_perm_scale),
        _stream(stream)), "moe_align_permute_noalloc")


def grouped_gemm_w13(p: Problem, x_perm, x_scale, w13, w13_scale, block_expert_ids,
                     num_post_padded, out, out_scale=None, fuse_act=False, stream=None):
    _check(lib().grouped_gemm_w13(
        _cp(p), _p(x_perm), _p(x_scale), _p(w13), _p(w13_scale), _p(block_expert_ids),
        _p(num_post_padded), _p(out), _p(out_scale), int(bool(fuse_act)), _stream(stream)),
        "grouped_gemm_w13")


def act_mul_quant(p: Problem, h1, num_post_padded, z, z_scale=None, stream=None):
    _check(lib().act_mul_quant(_cp(p), _p(h1), _p(num_post_padded), _p(z), _p(z_scale),
                               _stream(stream)), "act_mul_quant")


def grouped_gemm_w2(p: Problem, z, z_scale, w2, w2_scale, block_expert_ids, num_post_padded,
                    y2, stream=None):
    _check(lib().grouped_gemm_w2(_cp(p), _p(z), _p(z_scale), _p(w2), _p(w2_scale),
                                 _p(block_expert_ids), _p(num_post_padded), _p(y2),
                                 _stream(stream)), "grouped_gemm_w2")


def unpermute_reduce(p: Problem, y2, inv_perm, topk_weights, y, stream=None):
    _check(lib().unpermute_reduce(_cp(p), _p(y2), _p(inv_perm), _p(topk_weights), _p(y),
                                  _stream(stream)), "unpermute_reduce")


def grouped_gemm_w13_ex(p: Problem, x_perm, x_scale, w13, w13_scale, w13_bias, block_expert_ids,
                        num_post_padded, out, out_scale=None, fuse_act=False, stream=None):
    _check(lib().grouped_gemm_w13_ex(
        _cp(p), _p(x_perm), _p(x_scale), _p(w13), _p(w13_scale), _p(w13_bias),
        _p(block_expert_ids), _p(num_post_padded), _p(out), _p(out_scale), int(bool(fuse_act)),
        _stream(stream)), "grouped_gemm_w13_ex")


def grouped_gemm_w2_ex(p: Problem, z, z_scale, w2, w2_scale, w2_bias, block_expert_ids,
                       num_post_padded, sorted_ids, topk_weights, y2, stream=None):
    _check(lib().grouped_gemm_w2_ex(
        _cp(p), _p(z), _p(z_scale), _p(w2), _p(w2_scale), _p(w2_bias), _p(block_expert_ids),
        _p(num_post_padded), _p(sorted_ids), _p(topk_weights), _p(y2), _stream(stream)),
        "grouped_gemm_w2_ex")


def fused_experts_ex(p: Problem, x, w13, w13_scale, w13_bias, w2, w2_scale, w2_bias,
                     topk_weights, topk_ids, y, workspace, stream=None):
    _check(lib().fused_experts_ex(
        _cp(p), _p(x), _p(w13), _p(w13_scale), _p(w13_bias), _p(w2), _p(w2_scale), _p(w2_bias),
        _p(topk_weights), _p(topk_ids), _p(y), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)), "fused_experts_ex")


def moe_batched_workspace_bytes(p: Problem, max_tokens: int) -> int:
    return int(lib().moe_batched_workspace_bytes(_cp(p), int(max_tokens)))


def fused_experts_batched(p: Problem, x, expert_num_tokens, w13, w13_scale, w2, w2_scale, y,
                          workspace, expected_m=0, stream=None):
    """Expert MLPs on the batched layout x [E, max_tokens, H] (bf16) with
    per-expert counts (int32 [E]) into y of the same shape."""
    E, T, _ = x.shape
    _check(lib().fused_experts_batched(
        _cp(p), _p(x), _p(expert_num_tokens), int(T), int(expected_m), _p(w13), _p(w13_scale),
        _p(w2), _p(w2_scale), _p(y), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "fused_experts_batched")


SCORING = {"softmax": 0, "sigmoid": 1}


def moe_topk_router(logits, topk, topk_weights, topk_ids, token_expert_indices=None,
                    scoring="softmax", renormalize=True, expert_map=None, stream=None):
    """Router (softmax or sigmoid scores, top-k, optional renormalisation and
    expert map) into caller-allocated [M, topk] float32 / int32 tensors;
    logits [M, E] float32 or bfloat16, all on the device."""
    import torch
    M, E = logits.shape
    bf16 = logits.dtype == torch.bfloat16
    if not bf16 and logits.dtype != torch.float32:
        raise TypeError("logits must be float32 or bfloat16")
    _check(lib().moe_topk_router(int(M), int(E), int(topk), _p(logits), int(bf16),
                                 SCORING[scoring], int(bool(renormalize)), _p(expert_map),
                                 _p(topk_weights), _p(topk_ids), _p(token_expert_indices),
                                 _stream(stream)), "moe_topk_router")


def fused_experts(p: Problem, x, w13, w13_scale, w2, w2_scale, topk_weights, topk_ids, y,
                  workspace, stream=None):
    _check(lib().fused_experts(
        _cp(p), _p(x), _p(w13), _p(w13_scale), _p(w2), _p(w2_scale), _p(topk_weights),
        _p(topk_ids), _p(y), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "fused_experts")


def fused_experts_from_host(p: Problem, host_x, host_topk_ids, host_topk_weights, host_y,
                            w13, w13_scale, w2, w2_scale, workspace, stream=None):
    _check(lib().fused_experts_from_host(
        _cp(p), _p(host_x), _p(host_topk_ids), _p(host_topk_weights), _p(host_y), _p(w13),
        _p(w13_scale), _p(w2), _p(w2_scale), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)),
        "fused_experts_from_host")


def moe_gemm2_splits(p: Problem) -> int:
    return int(lib().moe_gemm2_splits(_cp(p)))


def moe_gemm2_partial_bytes(p: Problem, splits: int) -> int:
    return int(lib().moe_gemm2_partial_bytes(_cp(p), int(splits)))


def grouped_gemm_w2_split(p: Problem, z, w2, block_expert_ids, num_post_padded, sorted_ids,
                          splits, partial, stream=None):
    _check(lib().grouped_gemm_w2_split(
        _cp(p), _p(z), _p(w2), _p(block_expert_ids), _p(num_post_padded), _p(sorted_ids),
        int(splits), _p(partial), _stream(stream)), "grouped_gemm_w2_split")


def unpermute_reduce_split(p: Problem, partial, splits, inv_perm, topk_weights, y, stream=None):
    _check(lib().unpermute_reduce_split(
        _cp(p), _p(partial), int(splits), _p(inv_perm), _p(topk_weights), _p(y),
        _stream(stream)), "unpermute_reduce_split")


def moe_sync_status(stream=None) -> int:
    return int(lib().moe_sync_status(_stream(stream)))


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def moe_last_error_string() -> str:
    return lib().moe_last_error_string().decode()


def moe_debug_set_watchdog(limit_ns: int, never_arrive: bool = False):
    lib().moe_debug_set_watchdog(int(limit_ns), int(bool(never_arrive)))


BF16_GEMM_FORMS = {"auto": 0, "single": 1, "pairs": 2}


def moe_debug_set_bf16_gemm_form(form: str = "auto"):
    """Force the single-SM or the SM-pair bf16 GEMM (tests), or restore the
    size-based choice."""
    lib().moe_debug_set_bf16_gemm_form(BF16_GEMM_FORMS[form])


# ------------------------------------------------- buffer allocation helper
def stage_buffers(p: Problem, device="cuda"):
    """Allocates (torch.empty) the outputs of the staged entry points for
    problem ``p``, sized by the library's own bound; returns a dict."""
    import torch
    cap = moe_m_sum_bound(p)
    q = p.quant != "bf16"
    g = 32 if p.quant == "mxfp8" else 128      # activation quantisation group
    xb = torch.uint8 if q else torch.bfloat16
    i32 = dict(dtype=torch.int32, device=device)
    return {
        "sorted_ids": torch.empty(cap, **i32),
        "block_expert_ids": torch.empty(cap // p.block_size, **i32),
        "expert_offsets": torch.empty(p.E + 1, **i32),
        "num_post_padded": torch.empty(1, **i32),
        "inv_perm": torch.empty(p.M, p.topk, **i32),
        "x_perm": torch.empty(cap, p.H, dtype=xb, device=device),
        "x_perm_scale": torch.empty(cap, p.H // g, dtype=torch.float32, device=device)
        if q else None,
        "h1": torch.empty(cap, 2 * p.I, dtype=torch.bfloat16, device=device),
        "z": torch.empty(cap, p.I, dtype=xb, device=device),
        "z_scale": torch.empty(cap, p.I // g, dtype=torch.float32, device=device)
        if q else None,
        "y2": torch.empty(cap, p.H, dtype=torch.bfloat16, device=device),
        "y": torch.empty(p.M, p.H, dtype=torch.bfloat16, device=device),
        "align_ws": torch.empty(max(moe_align_workspace_bytes(p), 1), dtype=torch.uint8,
                                device=device),
    }
