"""Python binding of libob (include/ob.h): the GB300 implementation of the
error-compensated 1-bit compressed optimizer step (1-bit Adam / 1-bit
LAMB) and of the block-wise INT8 stochastic-rounding quantizer.

This module only marshals arguments: torch tensors become device pointers
and torch's current CUDA stream becomes the stream handle; every step of
the path runs in the CUDA kernels of libob.so.  There is no CPU fallback:
if libob.so is missing or cannot be loaded, `lib()` raises.

Two layers:
  * `ob_*` functions with the C names, taking an `ob_ctx` handle, tensors
    (or lists of tensors) and an optional stream;
  * `OneBitOptimizer`, which owns the device buffers of one simulated
    data-parallel job (W workers on one GPU) and calls the `ob_*` functions
    in the order of the method.
"""
import ctypes as ct
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libob.so")

OB_OK, OB_ERR_INVALID, OB_ERR_ALIGN, OB_ERR_UNSUPPORTED, OB_ERR_CUDA, OB_ERR_STATE = range(6)
OB_GRAD_F32, OB_GRAD_BF16 = 0, 1
OB_MODE_ADAM, OB_MODE_LAMB = 0, 1
OB_MAX_WORKERS = 64
OB_NOALLOC_SCRATCH_BYTES = 4 << 20  # the static scratch of ob_compress_noalloc
OB_FLAG_NO_RATIO_EF = 1 << 0
OB_FLAG_FROZEN_C = 1 << 1

# Every entry point include/ob.h declares.
EXPORTS = (
    "ob_init", "ob_destroy", "ob_last_error", "ob_get_layout", "ob_workspace_bytes",
    "ob_set_workspace", "ob_warmup_step", "ob_begin_compression", "ob_compress",
    "ob_server_reduce", "ob_decompress", "ob_adam_step", "ob_lamb_step", "ob_step",
    "ob_materialize_errors", "ob_device_error", "ob_quant_int8", "ob_compress_noalloc",
    "ob_compress_signm", "ob_reset_errors", "ob_quant_int8_ef",
    "ob_qb_sizes", "ob_zero_errors", "ob_compress_qb", "ob_server_reduce_qb", "ob_adam_step_qb",
    "ob_compress_f16", "ob_server_reduce_f16", "ob_adam_step_f16",
    "ob_compress_signm_ls", "ob_server_reduce_db", "ob_lamb_step_signm", "ob_step_db",
    "ob_noalloc_device_error", "ob_error_norm", "ob_plan_step", "ob_codec_step",
    "ob_compress_worker", "ob_server_reduce_part", "ob_reset_errors_rank",
)


class OBError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"libob status {status}: {msg}")
        self.status = status


class ob_config(ct.Structure):
    _fields_ = [("n", ct.c_size_t), ("W", ct.c_int), ("chunk", ct.c_size_t),
                ("align", ct.c_size_t), ("grad_dtype", ct.c_int), ("n_layers", ct.c_int),
                ("layer_offsets", ct.POINTER(ct.c_size_t)),
                ("b1", ct.c_float), ("b2", ct.c_float), ("eps", ct.c_float),
                ("lr", ct.c_float), ("r_thr", ct.c_float), ("r_min", ct.c_float),
                ("r_max", ct.c_float), ("c_min", ct.c_float), ("c_max", ct.c_float),
                ("flags", ct.c_uint32), ("clip_value", ct.c_float),
                ("reset_interval", ct.c_uint32), ("send_period", ct.c_uint32),
                ("seed", ct.c_uint64)]


class ob_layout(ct.Structure):
    _fields_ = [("n", ct.c_size_t), ("n_pad", ct.c_size_t), ("P", ct.c_size_t),
                ("chunk", ct.c_size_t), ("chunks_per_partition", ct.c_size_t),
                ("n_chunks", ct.c_size_t), ("words_per_worker", ct.c_size_t),
                ("n_tiles", ct.c_size_t), ("W", ct.c_int), ("n_layers", ct.c_int)]


class ob_plan(ct.Structure):
    _fields_ = [("reset", ct.c_int), ("send", ct.c_int), ("key", ct.c_uint64),
                ("step", ct.c_uint64)]


class ob_layer_state(ct.Structure):
    _fields_ = [(k, ct.c_void_p) for k in
                ("s", "c_avg", "r_prev", "c_prev", "c_prev2", "c_sum", "c_t")]


_lib = None


def lib():
    """Loads libob.so (built by __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                "g.build()'` (nvcc, sm_103a); there is no CPU fallback")
        L = ct.CDLL(LIB_PATH)
        vp, sz, i32, u64 = ct.c_void_p, ct.c_size_t, ct.c_int, ct.c_uint64
        L.ob_init.argtypes = [ct.POINTER(ob_config), ct.POINTER(vp)]
        L.ob_destroy.argtypes = [vp]
        L.ob_last_error.argtypes = [vp]
        L.ob_last_error.restype = ct.c_char_p
        L.ob_get_layout.argtypes = [vp, ct.POINTER(ob_layout)]
        L.ob_workspace_bytes.argtypes = [vp, ct.POINTER(sz)]
        L.ob_set_workspace.argtypes = [vp, vp, sz, vp]
        L.ob_warmup_step.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp]
        L.ob_begin_compression.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp]
        L.ob_compress.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        L.ob_server_reduce.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        L.ob_decompress.argtypes = [vp, vp, vp, vp, vp, vp]
        L.ob_adam_step.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        L.ob_lamb_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.ob_step.argtypes = [vp] * 14
        L.ob_materialize_errors.argtypes = [vp] * 8
        L.ob_device_error.argtypes = [vp, ct.POINTER(ct.c_uint), vp]
        L.ob_quant_int8.argtypes = [vp, sz, vp, vp, u64, u64, vp, vp]
        L.ob_compress_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        L.ob_noalloc_device_error.argtypes = [ct.POINTER(ct.c_uint), vp]
        L.ob_error_norm.argtypes = [vp] * 9
        L.ob_plan_step.argtypes = [vp, i32, u64, ct.POINTER(ob_plan)]
        L.ob_codec_step.argtypes = [vp, i32, u64] + [vp] * 11
        L.ob_compress_worker.argtypes = [vp] * 10
        L.ob_server_reduce_part.argtypes = [vp, i32] + [vp] * 7
        L.ob_reset_errors_rank.argtypes = [vp, i32] + [vp] * 7
        L.ob_compress_signm.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        L.ob_reset_errors.argtypes = [vp] * 8
        L.ob_quant_int8_ef.argtypes = [vp, vp, sz, vp, vp, u64, u64, vp, vp, vp]
        L.ob_qb_sizes.argtypes = [vp, i32, ct.POINTER(sz), ct.POINTER(sz)]
        L.ob_zero_errors.argtypes = [vp, vp, vp, vp]
        L.ob_compress_qb.argtypes = [vp, i32, vp, vp, vp, vp, vp, u64, u64, vp]
        L.ob_server_reduce_qb.argtypes = [vp, i32, vp, vp, vp, vp, vp, u64, u64, vp]
        L.ob_adam_step_qb.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
        L.ob_compress_f16.argtypes = [vp, i32, vp, vp, vp, vp, vp]
        L.ob_server_reduce_f16.argtypes = [vp, vp, vp, vp, vp]
        L.ob_adam_step_f16.argtypes = [vp, i32, vp, vp, vp, vp, vp]
        L.ob_compress_signm_ls.argtypes = [vp] * 9
        L.ob_server_reduce_db.argtypes = [vp] * 10
        L.ob_lamb_step_signm.argtypes = [vp] * 10
        L.ob_step_db.argtypes = [vp] * 15
        for name in EXPORTS:
            if name != "ob_last_error":
                getattr(L, name).restype = ct.c_int
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
# Marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(x):
    """Device (or host) address of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptr_array(xs):
    arr = (ct.c_void_p * len(xs))(*[_ptr(x) for x in xs])
    return arr


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, ctx=None):
    if status != OB_OK:
        msg = lib().ob_last_error(ctx).decode(errors="replace")
        raise OBError(status, msg)


class LayerState:
    """Per-layer 1-bit LAMB state: seven float32 device tensors of n_layers
    entries (s, c_avg, r_prev, c_prev, c_prev2, c_sum, c_t)."""

    FIELDS = ("s", "c_avg", "r_prev", "c_prev", "c_prev2", "c_sum", "c_t")

    def __init__(self, n_layers, device="cuda"):
        import torch
        for f in self.FIELDS:
            setattr(self, f, torch.zeros(n_layers, dtype=torch.float32, device=device))

    def struct(self):
        return ob_layer_state(*[_ptr(getattr(self, f)) for f in self.FIELDS])


def _ls(ls):
    if ls is None:
        return None
    return ct.byref(ls.struct() if isinstance(ls, LayerState) else ls)


# ---------------------------------------------------------------------------
# The C entry points, same names
# ---------------------------------------------------------------------------

def ob_init(n, W, chunk, align=4096, grad_dtype=OB_GRAD_F32, layer_offsets=None,
            b1=0.9, b2=0.999, eps=1e-8, lr=1e-4, r_thr=0.1, r_min=0.5, r_max=4.0,
            c_min=0.01, c_max=10.0, flags=0, clip_value=0.0, reset_interval=0, send_period=0,
            seed=0):
    """Returns an opaque ctx handle (int).  layer_offsets: sequence of
    n_layers+1 ints, or None for one layer.  reset_interval, send_period and
    seed configure the schedules of ob_plan_step."""
    cfg = ob_config(n=n, W=W, chunk=chunk, align=align, grad_dtype=grad_dtype,
                    b1=b1, b2=b2, eps=eps, lr=lr, r_thr=r_thr, r_min=r_min, r_max=r_max,
                    c_min=c_min, c_max=c_max, flags=flags, clip_value=clip_value,
                    reset_interval=reset_interval, send_period=send_period, seed=seed)
    keep = None
    if layer_offsets is not None:
        keep = (ct.c_size_t * len(layer_offsets))(*[int(x) for x in layer_offsets])
        cfg.n_layers = len(layer_offsets) - 1
        cfg.layer_offsets = ct.cast(keep, ct.POINTER(ct.c_size_t))
    h = ct.c_void_p()
    _check(lib().ob_init(ct.byref(cfg), ct.byref(h)))
    return h.value


def ob_destroy(ctx):
    """Frees the host context (device buffers stay the caller's)."""
    lib().ob_destroy(ctx)


def ob_last_error(ctx=None):
    """The context's last error message (or the global one for ctx None)."""
    return lib().ob_last_error(ctx).decode(errors="replace")


def ob_get_layout(ctx):
    """The layout of the fused buffer as a dict (n_pad, P, chunk, n_chunks, words_per_worker, n_tiles, ...)."""
    lay = ob_layout()
    _check(lib().ob_get_layout(ctx, ct.byref(lay)), ctx)
    return {k: getattr(lay, k) for k, _ in ob_layout._fields_}


def ob_workspace_bytes(ctx):
    """Bytes of device scratch the context needs (tile partials, per-layer tables)."""
    b = ct.c_size_t()
    _check(lib().ob_workspace_bytes(ctx, ct.byref(b)), ctx)
    return b.value


def ob_set_workspace(ctx, workspace, nbytes=None, stream=None):
    """Hands the context its device scratch and enqueues its initialisation on `stream`."""
    if nbytes is None:
        nbytes = workspace.numel() * workspace.element_size()
    _check(lib().ob_set_workspace(ctx, _ptr(workspace), nbytes, _stream(stream)), ctx)


def ob_warmup_step(ctx, grads, m, v, p, mode=OB_MODE_ADAM, ls=None, stream=None):
    """One uncompressed warmup step of 1-bit Adam (mode ADAM) or 1-bit LAMB (mode LAMB, with ls)."""
    _check(lib().ob_warmup_step(ctx, _ptr_array(grads), _ptr(m), _ptr(v), _ptr(p), mode,
                                _ls(ls), _stream(stream)), ctx)


def ob_begin_compression(ctx, err, err_s, bits, scales, sbits, sscales, m=None, v=None,
                         v_fresh=None, ls=None, warmup_steps=0, stream=None):
    """End of warmup: zeroes errors and sign buffers, freezes v; for LAMB sets sigma, c_avg and the coefficient history."""
    _check(lib().ob_begin_compression(ctx, None if err is None else _ptr_array(err),
                                      _ptr(err_s), _ptr(bits),
                                      _ptr(scales), _ptr(sbits), _ptr(sscales), _ptr(m),
                                      _ptr(v), _ptr(v_fresh), _ls(ls), warmup_steps,
                                      _stream(stream)), ctx)


def ob_compress(ctx, grads, m, err, bits, scales, ls=None, stream=None):
    """Worker compression of all W workers with the dense momentum m (LAMB if ls is given)."""
    _check(lib().ob_compress(ctx, _ptr_array(grads), _ptr(m), _ptr_array(err), _ptr(bits),
                             _ptr(scales), _ls(ls), _stream(stream)), ctx)


def ob_compress_noalloc(ctx, grads, m, err, bits, scales, stream=None):
    """ob_compress (1-bit Adam) with the library's static scratch instead of
    a workspace: for callers that cannot allocate device memory."""
    _check(lib().ob_compress_noalloc(ctx, _ptr_array(grads), _ptr(m), _ptr_array(err),
                                     _ptr(bits), _ptr(scales), _stream(stream)), ctx)


def ob_noalloc_device_error(stream=None):
    """Reads and clears the error word of ob_compress_noalloc's static scratch
    on the current device (0 = none)."""
    v = ct.c_uint()
    _check(lib().ob_noalloc_device_error(ct.byref(v), _stream(stream)))
    return v.value


def ob_compress_signm(ctx, grads, sbits, sscales, err, bits, scales, stream=None):
    """ob_compress for 1-bit Adam reading the momentum as sscale*sign(sbit)."""
    _check(lib().ob_compress_signm(ctx, _ptr_array(grads), _ptr(sbits), _ptr(sscales),
                                   _ptr_array(err), _ptr(bits), _ptr(scales), _stream(stream)),
           ctx)


def ob_compress_signm_ls(ctx, grads, sbits, sscales, err, bits, scales, ls=None, stream=None):
    """ob_compress_signm for 1-bit Adam (ls None) or 1-bit LAMB, the momentum
    read as sscale*sign(sbit) (/ sigma_l for LAMB)."""
    _check(lib().ob_compress_signm_ls(ctx, _ptr_array(grads), _ptr(sbits), _ptr(sscales),
                                      _ptr_array(err), _ptr(bits), _ptr(scales), _ls(ls),
                                      _stream(stream)), ctx)


def ob_server_reduce_db(ctx, bits, scales, err_s, sbits_old, sscales_old, sbits, sscales,
                        ls=None, stream=None):
    """ob_server_reduce decoding e_s with (sbits_old, sscales_old) and writing
    the new words and scales to (sbits, sscales)."""
    _check(lib().ob_server_reduce_db(ctx, _ptr(bits), _ptr(scales), _ptr(err_s),
                                     _ptr(sbits_old), _ptr(sscales_old), _ptr(sbits),
                                     _ptr(sscales), _ls(ls), _stream(stream)), ctx)


def ob_lamb_step_signm(ctx, sbits_prev, sscales_prev, sbits, sscales, v_frozen, v_fresh, p, ls,
                       stream=None):
    """ob_lamb_step with m_{t-1} and m_t read from the previous and the
    current server output; no dense m."""
    _check(lib().ob_lamb_step_signm(ctx, _ptr(sbits_prev), _ptr(sscales_prev), _ptr(sbits),
                                    _ptr(sscales), _ptr(v_frozen), _ptr(v_fresh), _ptr(p),
                                    _ls(ls), _stream(stream)), ctx)


def ob_step_db(ctx, grads, err, bits, scales, err_s, sbits_prev, sscales_prev, sbits, sscales,
               v_frozen, v_fresh, p, ls=None, stream=None):
    """One compressed step, momentum in sign form, server output
    double-buffered: reads (sbits_prev, sscales_prev), writes (sbits, sscales)."""
    _check(lib().ob_step_db(ctx, _ptr_array(grads), _ptr_array(err), _ptr(bits), _ptr(scales),
                            _ptr(err_s), _ptr(sbits_prev), _ptr(sscales_prev), _ptr(sbits),
                            _ptr(sscales), _ptr(v_frozen), _ptr(v_fresh), _ptr(p), _ls(ls),
                            _stream(stream)), ctx)


def ob_server_reduce(ctx, bits, scales, err_s, sbits, sscales, ls=None, stream=None):
    """Server average of the workers' chunks, plus its own error, compressed again (in place)."""
    _check(lib().ob_server_reduce(ctx, _ptr(bits), _ptr(scales), _ptr(err_s), _ptr(sbits),
                                  _ptr(sscales), _ls(ls), _stream(stream)), ctx)


def ob_decompress(ctx, sbits, sscales, out, ls=None, stream=None):
    """out = sscale*sign(sbit) (over sigma_l with ls); padding 0."""
    _check(lib().ob_decompress(ctx, _ptr(sbits), _ptr(sscales), _ls(ls), _ptr(out),
                               _stream(stream)), ctx)


def ob_adam_step(ctx, sbits, sscales, v_frozen, m, p, stream=None):
    """Unpack + frozen-variance Adam update; m None keeps the momentum in sign form."""
    _check(lib().ob_adam_step(ctx, _ptr(sbits), _ptr(sscales), _ptr(v_frozen), _ptr(m),
                              _ptr(p), _stream(stream)), ctx)


def ob_lamb_step(ctx, sbits, sscales, v_frozen, v_fresh, m, p, ls, stream=None):
    """Unpack + 1-bit LAMB update (passes A and B) with the dense momentum m."""
    _check(lib().ob_lamb_step(ctx, _ptr(sbits), _ptr(sscales), _ptr(v_frozen), _ptr(v_fresh),
                              _ptr(m), _ptr(p), _ls(ls), _stream(stream)), ctx)


def ob_step(ctx, grads, m, err, bits, scales, err_s, sbits, sscales, v_frozen, v_fresh, p,
            ls=None, stream=None):
    """compress + server_reduce + update in one call; m None (1-bit Adam) uses the sign-form momentum."""
    _check(lib().ob_step(ctx, _ptr_array(grads), _ptr(m), _ptr_array(err), _ptr(bits),
                         _ptr(scales), _ptr(err_s), _ptr(sbits), _ptr(sscales),
                         _ptr(v_frozen), _ptr(v_fresh), _ptr(p), _ls(ls), _stream(stream)),
           ctx)


def ob_materialize_errors(ctx, err, bits, scales, err_s, sbits, sscales, stream=None):
    """Writes the true errors e' into err and err_s and zeroes the scales (checkpoint form)."""
    _check(lib().ob_materialize_errors(ctx, _ptr_array(err), _ptr(bits), _ptr(scales),
                                       _ptr(err_s), _ptr(sbits), _ptr(sscales),
                                       _stream(stream)), ctx)


def ob_reset_errors(ctx, err, bits, scales, err_s, sbits, sscales, stream=None):
    """Periodic error reset: the next compression sees worker and server errors of 0."""
    _check(lib().ob_reset_errors(ctx, _ptr_array(err), _ptr(bits), _ptr(scales), _ptr(err_s),
                                 _ptr(sbits), _ptr(sscales), _stream(stream)), ctx)


def ob_error_norm(ctx, err, bits, scales, err_s, sbits, sscales, out, stream=None):
    """Per chunk, the sums of squares of every worker's and the server's
    true error (the 1-bit error monitor): out has (W+1)*n_chunks floats."""
    _check(lib().ob_error_norm(ctx, _ptr_array(err), _ptr(bits), _ptr(scales), _ptr(err_s),
                               _ptr(sbits), _ptr(sscales), _ptr(out), _stream(stream)), ctx)


def ob_plan_step(ctx, bits, t):
    """The schedule of compressed step t (from 1) for a group of width bits:
    a dict with reset, send, key and step (host only)."""
    pl = ob_plan()
    _check(lib().ob_plan_step(ctx, bits, t, ct.byref(pl)), ctx)
    return {"reset": bool(pl.reset), "send": bool(pl.send), "key": pl.key, "step": pl.step}


def ob_codec_step(ctx, bits, t, grads, m, err, msg, msg_scales, err_s, smsg, smsg_scales,
                  v_frozen, p, stream=None):
    """One compressed step of a codec group (bits 2, 4, 8 or 16) at
    compressed step t, with the schedule of ob_plan_step applied inside."""
    _check(lib().ob_codec_step(ctx, bits, t, _ptr_array(grads), _ptr(m), _ptr_array(err),
                               _ptr(msg), _ptr(msg_scales), _ptr(err_s), _ptr(smsg),
                               _ptr(smsg_scales), _ptr(v_frozen), _ptr(p), _stream(stream)),
           ctx)


def ob_compress_worker(ctx, grad, err, bits_row, scales_row, m=None, msbits=None,
                       msscales=None, ls=None, stream=None):
    """One rank's compression of its own worker (dense m, or the momentum
    in sign form from the gathered server output)."""
    _check(lib().ob_compress_worker(ctx, _ptr(grad), _ptr(m), _ptr(msbits), _ptr(msscales),
                                    _ptr(err), _ptr(bits_row), _ptr(scales_row), _ls(ls),
                                    _stream(stream)), ctx)


def ob_server_reduce_part(ctx, j, recv_bits, recv_scales, err_s_part, sbits_part,
                          sscales_part, ls=None, stream=None):
    """One rank's server: partition j from the W received blocks."""
    _check(lib().ob_server_reduce_part(ctx, j, _ptr(recv_bits), _ptr(recv_scales),
                                       _ptr(err_s_part), _ptr(sbits_part), _ptr(sscales_part),
                                       _ls(ls), _stream(stream)), ctx)


def ob_reset_errors_rank(ctx, j, err, bits_row, scales_row, err_s_part, sbits_part,
                         sscales_part, stream=None):
    """One rank's periodic error reset: its own worker error and its server
    partition's error become 0 (deferred form; words and scales untouched)."""
    _check(lib().ob_reset_errors_rank(ctx, j, _ptr(err), _ptr(bits_row), _ptr(scales_row),
                                      _ptr(err_s_part), _ptr(sbits_part), _ptr(sscales_part),
                                      _stream(stream)), ctx)


def ob_device_error(ctx, stream=None):
    """Reads and clears the device error word (0 = none)."""
    v = ct.c_uint()
    _check(lib().ob_device_error(ctx, ct.byref(v), _stream(stream)), ctx)
    return v.value


def ob_quant_int8(g, q, block_scales, seed, step, deq=None, n=None, stream=None):
    """Block-256 INT8 stochastic-rounding quantizer of g (Philox4x32-10 uniforms)."""
    if n is None:
        n = g.numel()
    _check(lib().ob_quant_int8(_ptr(g), n, _ptr(q), _ptr(block_scales), seed, step, _ptr(deq),
                               _stream(stream)))


def ob_quant_int8_ef(g, e, q, block_scales, seed, step, deq=None, block_err2=None, n=None,
                     stream=None):
    """INT8 quantizer with error feedback (e updated) and the per-block error monitor."""
    if n is None:
        n = g.numel()
    _check(lib().ob_quant_int8_ef(_ptr(g), _ptr(e), n, _ptr(q), _ptr(block_scales), seed, step,
                                  _ptr(deq), _ptr(block_err2), _stream(stream)))


def ob_qb_sizes(ctx, bits):
    """(words_per_worker, n_blocks) of the b-bit codec."""
    w, b = ct.c_size_t(), ct.c_size_t()
    _check(lib().ob_qb_sizes(ctx, bits, ct.byref(w), ct.byref(b)), ctx)
    return w.value, b.value


def ob_zero_errors(ctx, err, err_s, stream=None):
    """Zeroes a codec group's worker and server errors (start of compression)."""
    _check(lib().ob_zero_errors(ctx, _ptr_array(err), _ptr(err_s), _stream(stream)), ctx)


def ob_compress_qb(ctx, bits, grads, m, err, codes, bscales, seed, step, stream=None):
    """Worker compression with the b-bit block codec (b = 2, 4, 8)."""
    _check(lib().ob_compress_qb(ctx, bits, _ptr_array(grads), _ptr(m), _ptr_array(err),
                                _ptr(codes), _ptr(bscales), seed, step, _stream(stream)), ctx)


def ob_server_reduce_qb(ctx, bits, codes, bscales, err_s, scodes, sbscales, seed, step,
                        stream=None):
    """Server average and re-quantisation with the b-bit block codec."""
    _check(lib().ob_server_reduce_qb(ctx, bits, _ptr(codes), _ptr(bscales), _ptr(err_s),
                                     _ptr(scodes), _ptr(sbscales), seed, step, _stream(stream)),
           ctx)


def ob_adam_step_qb(ctx, bits, scodes, sbscales, v_frozen, m, p, stream=None):
    """Decode of the server's b-bit message + frozen-variance Adam."""
    _check(lib().ob_adam_step_qb(ctx, bits, _ptr(scodes), _ptr(sbscales), _ptr(v_frozen), _ptr(m),
                                 _ptr(p), _stream(stream)), ctx)


def ob_compress_f16(ctx, send, grads, m, err, h, stream=None):
    """Worker step of the FP16 codec (sent only when `send`)."""
    _check(lib().ob_compress_f16(ctx, int(bool(send)), _ptr_array(grads), _ptr(m),
                                 _ptr_array(err), _ptr(h), _stream(stream)), ctx)


def ob_server_reduce_f16(ctx, h, err_s, hs, stream=None):
    """Server average of the FP16 messages, rounded to FP16 with error feedback."""
    _check(lib().ob_server_reduce_f16(ctx, _ptr(h), _ptr(err_s), _ptr(hs), _stream(stream)), ctx)


def ob_adam_step_f16(ctx, send, hs, v_frozen, m, p, stream=None):
    """Adam update from the FP16 server message (m = 0, p unchanged when not sent)."""
    _check(lib().ob_adam_step_f16(ctx, int(bool(send)), _ptr(hs), _ptr(v_frozen), _ptr(m),
                                  _ptr(p), _stream(stream)), ctx)


# ---------------------------------------------------------------------------
# One simulated data-parallel job
# ---------------------------------------------------------------------------

class OneBitOptimizer:
    """Device buffers and call order of one 1-bit Adam / 1-bit LAMB job with
    W workers simulated on one GPU.

    Buffers (torch, on `device`): m, v (frozen after warmup), p, v_fresh
    (LAMB), err[W], err_s, bits [W, words], scales [W, n_chunks], sbits,
    sscales, the workspace, and the per-layer LAMB state."""

    def __init__(self, n, W, chunk, align=4096, grad_dtype="f32", layer_offsets=None,
                 lamb=False, device="cuda", sign_momentum=False, reset_interval=0, **hp):
        """sign_momentum: after the first compressed step the momentum is
        held as (sbits, sscales) -- exactly sscale*sign, over sigma_l for
        LAMB -- and the dense m buffer is only refreshed by materialize_m().
        With LAMB the server output is double-buffered (the update reads
        the previous step's words too): sbits/sscales always name the last
        step's output, sbits_alt/sscales_alt the other pair.
        reset_interval > 0: before every reset_interval-th compressed step
        the worker and server errors are reset to 0 (ob_reset_errors).
        hp may hold clip_value (> 0: clamp of the compensated values)."""
        import torch
        self.lamb = lamb
        self.reset_interval = reset_interval
        self.cstep = 0
        self.sign_momentum = sign_momentum
        self.m_in_signs = False
        self.grad_dtype = grad_dtype
        self.ctx = ob_init(n, W, chunk, align,
                           OB_GRAD_BF16 if grad_dtype == "bf16" else OB_GRAD_F32,
                           layer_offsets, reset_interval=reset_interval, **hp)
        lay = ob_get_layout(self.ctx)
        self.layout = lay
        self.n, self.W, self.n_pad = n, W, lay["n_pad"]
        z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=device)
        self.m, self.v, self.p = z(self.n_pad), z(self.n_pad), z(self.n_pad)
        self.v_fresh = z(self.n_pad) if lamb else None
        self.err = [z(self.n_pad) for _ in range(W)]
        self.err_s = z(self.n_pad)
        words = lay["words_per_worker"]
        self.bits = z(W, words, dt=torch.int32)
        self.scales = z(W, lay["n_chunks"])
        self.sbits = z(words, dt=torch.int32)
        self.sscales = z(lay["n_chunks"])
        self.double_buffered = bool(sign_momentum and lamb)
        self.sbits_alt = z(words, dt=torch.int32) if self.double_buffered else None
        self.sscales_alt = z(lay["n_chunks"]) if self.double_buffered else None
        nbytes = ob_workspace_bytes(self.ctx)
        self.workspace = torch.zeros((nbytes + 255) // 256 * 256 // 4, dtype=torch.float32,
                                     device=device)
        ob_set_workspace(self.ctx, self.workspace, nbytes)
        self.ls = LayerState(lay["n_layers"], device) if lamb else None
        self.warmup_steps = 0

    def close(self):
        if self.ctx:
            ob_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def grad_buffers(self):
        import torch
        dt = torch.bfloat16 if self.grad_dtype == "bf16" else torch.float32
        return [torch.zeros(self.n_pad, dtype=dt, device=self.m.device) for _ in range(self.W)]

    def warmup_step(self, grads, stream=None):
        ob_warmup_step(self.ctx, grads, self.m, self.v, self.p,
                       OB_MODE_LAMB if self.lamb else OB_MODE_ADAM, self.ls, stream)
        self.warmup_steps += 1

    def begin_compression(self, stream=None):
        ob_begin_compression(self.ctx, self.err, self.err_s, self.bits, self.scales, self.sbits,
                             self.sscales, self.m, self.v, self.v_fresh,
                             self.ls if self.lamb else None, max(self.warmup_steps, 1), stream)
        self.m_in_signs = False
        self.cstep = 0

    def reset_errors(self, stream=None):
        ob_reset_errors(self.ctx, self.err, self.bits, self.scales, self.err_s, self.sbits,
                        self.sscales, stream)

    def compressed_step(self, grads, stream=None):
        if self.reset_interval and ob_plan_step(self.ctx, 1, self.cstep + 1)["reset"]:
            self.reset_errors(stream)
        self.cstep += 1
        if self.double_buffered and self.m_in_signs:
            self._step_db(grads, stream)
            return
        m = None if self.m_in_signs else self.m
        ob_step(self.ctx, grads, m, self.err, self.bits, self.scales, self.err_s,
                self.sbits, self.sscales, self.v, self.v_fresh, self.p,
                self.ls if self.lamb else None, stream)
        if self.sign_momentum and not self.m_in_signs:
            self.m_in_signs = True  # the next steps read the momentum from the signs

    def _step_db(self, grads, stream=None):
        """One double-buffered sign-form step; the new output becomes
        (sbits, sscales)."""
        ob_step_db(self.ctx, grads, self.err, self.bits, self.scales, self.err_s,
                   self.sbits, self.sscales, self.sbits_alt, self.sscales_alt, self.v,
                   self.v_fresh, self.p, self.ls if self.lamb else None, stream)
        self._swap()

    def _swap(self):
        self.sbits, self.sbits_alt = self.sbits_alt, self.sbits
        self.sscales, self.sscales_alt = self.sscales_alt, self.sscales

    def capture_step(self, grads):
        """Captures one compressed step on the gradient buffers `grads` into
        a CUDA graph and returns an object whose replay() runs that step
        with whatever the buffers hold -- one launch instead of five or six,
        for sizes where launches dominate.  The step reads every per-step
        quantity (scales, sign words, LAMB state) from device memory, so
        replays are the same steps as eager calls.  Host-side schedules are
        not replayed: capture after the first compressed step when the
        momentum is held in sign form, and without reset_interval; replay()
        refuses to run once the momentum's form has changed since the
        capture (materialize_m / materialize_errors).  The library
        allocates nothing, so capture needs no memory pool."""
        import torch
        if self.reset_interval:
            raise ValueError("capture_step: reset_interval is a host-side schedule")
        if self.sign_momentum and not self.m_in_signs:
            raise ValueError("capture_step: take the first compressed step eagerly")
        if self.double_buffered:
            return _AlternatingGraphs(self, grads)
        graph = torch.cuda.CUDAGraph()
        m = None if self.m_in_signs else self.m
        with torch.cuda.graph(graph):
            ob_step(self.ctx, grads, m, self.err, self.bits, self.scales, self.err_s,
                    self.sbits, self.sscales, self.v, self.v_fresh, self.p,
                    self.ls if self.lamb else None)
        return _StepGraph(self, graph)

    def error_norm(self, out=None, stream=None):
        """The 1-bit error monitor: a (W+1, n_chunks) float32 tensor whose
        row w (and row W, the server's) holds, per chunk, the sum of the
        squared true errors after the last step."""
        import torch
        if out is None:
            out = torch.empty((self.W + 1, self.layout["n_chunks"]), dtype=torch.float32,
                              device=self.m.device)
        ob_error_norm(self.ctx, self.err, self.bits, self.scales, self.err_s, self.sbits,
                      self.sscales, out, stream)
        return out

    def materialize_m(self, stream=None):
        """Writes the dense momentum (it is exact: sscale*sign)."""
        if self.m_in_signs:
            ob_decompress(self.ctx, self.sbits, self.sscales, self.m,
                          self.ls if self.lamb else None, stream)
            self.m_in_signs = False

    def materialize_errors(self, stream=None):
        self.materialize_m(stream)  # the sign form is lost once sscales are cleared
        ob_materialize_errors(self.ctx, self.err, self.bits, self.scales, self.err_s,
                              self.sbits, self.sscales, stream)


class _StepGraph:
    """A captured compressed step: replay() runs it if the optimizer still
    holds its momentum in the form the capture recorded."""

    def __init__(self, opt, graph):
        self.opt, self.graph, self.m_in_signs = opt, graph, opt.m_in_signs

    def _check(self):
        if self.opt.m_in_signs != self.m_in_signs:
            raise RuntimeError("replay: the momentum's form changed since the capture; "
                               "capture the step again")

    def replay(self):
        self._check()
        self.graph.replay()


class _AlternatingGraphs(_StepGraph):
    """Two CUDA graphs of one double-buffered sign-form step, one for each
    orientation of the two server buffers; replay() runs the one that
    matches the optimizer's current buffers and swaps them, so replays are
    the same steps as eager calls."""

    def __init__(self, opt, grads):
        import torch
        super().__init__(opt, None)
        self.graphs = {}
        for _ in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                ob_step_db(opt.ctx, grads, opt.err, opt.bits, opt.scales, opt.err_s,
                           opt.sbits, opt.sscales, opt.sbits_alt, opt.sscales_alt, opt.v,
                           opt.v_fresh, opt.p, opt.ls if opt.lamb else None)
            self.graphs[opt.sbits.data_ptr()] = g
            opt._swap()  # capture only records; the other orientation next

    def replay(self):
        self._check()
        self.graphs[self.opt.sbits.data_ptr()].replay()
        self.opt._swap()


class CodecGroup:
    """One group of layerwise mixed widths compressed with the b-bit codec
    (bits 2, 4, 8) or the FP16 codec (bits 16, exchanged on every
    `period`-th compressed step), with 1-bit Adam's frozen-variance update.
    Buffers: m, v, p, err[W], err_s, and the messages (codes/bscales and
    scodes/sbscales, or h and hs)."""

    def __init__(self, n, W, bits, align=4096, grad_dtype="f32", device="cuda", period=10,
                 seed=1234, reset_interval=0, **hp):
        import torch
        if bits not in (2, 4, 8, 16):
            raise ValueError(f"bits = {bits}: the codec groups take 2, 4, 8 or 16")
        self.bits, self.period, self.seed = bits, period, seed
        self.reset_interval = reset_interval
        self.grad_dtype = grad_dtype
        self.ctx = ob_init(n, W, align, align,
                           OB_GRAD_BF16 if grad_dtype == "bf16" else OB_GRAD_F32, None,
                           reset_interval=reset_interval, send_period=period, seed=seed, **hp)
        lay = ob_get_layout(self.ctx)
        self.layout = lay
        self.n, self.W, self.n_pad = n, W, lay["n_pad"]
        z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=device)
        self.m, self.v, self.p = z(self.n_pad), z(self.n_pad), z(self.n_pad)
        self.err = [z(self.n_pad) for _ in range(W)]
        self.err_s = z(self.n_pad)
        if bits == 16:
            self.h = z(W, self.n_pad, dt=torch.int16)
            self.hs = z(self.n_pad, dt=torch.int16)
        else:
            words, nblk = ob_qb_sizes(self.ctx, bits)
            self.codes = z(W, words, dt=torch.int32)
            self.bscales = z(W, nblk)
            self.scodes = z(words, dt=torch.int32)
            self.sbscales = z(nblk)
        nbytes = ob_workspace_bytes(self.ctx)  # the warmup step's scratch
        self.workspace = torch.zeros((nbytes + 255) // 256 * 256 // 4, dtype=torch.float32,
                                     device=device)
        ob_set_workspace(self.ctx, self.workspace, nbytes)
        self.t = 0

    def close(self):
        if self.ctx:
            ob_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def grad_buffers(self):
        import torch
        dt = torch.bfloat16 if self.grad_dtype == "bf16" else torch.float32
        return [torch.zeros(self.n_pad, dtype=dt, device=self.m.device) for _ in range(self.W)]

    def warmup_step(self, grads, stream=None):
        ob_warmup_step(self.ctx, grads, self.m, self.v, self.p, OB_MODE_ADAM, None, stream)

    def begin_compression(self, stream=None):
        ob_zero_errors(self.ctx, self.err, self.err_s, stream)
        self.t = 0

    @property
    def key(self):
        """The Philox key the library uses for this group (seed + bits)."""
        return ob_plan_step(self.ctx, self.bits, 1)["key"]

    def compressed_step(self, grads, stream=None):
        self.t += 1
        if self.bits == 16:
            ob_codec_step(self.ctx, 16, self.t, grads, self.m, self.err, self.h, None,
                          self.err_s, self.hs, None, self.v, self.p, stream)
        else:
            ob_codec_step(self.ctx, self.bits, self.t, grads, self.m, self.err, self.codes,
                          self.bscales, self.err_s, self.scodes, self.sbscales, self.v, self.p,
                          stream)


class MixedOptimizer:
    """Layerwise mixed bit widths: one group per width, each a fused buffer
    of its own (the "1bit Adam" write-up's §3.2 table: 1 bit for embeddings
    and dense layers, 2 for convolution weights, FP16 every 10th step for
    normalisation parameters).  `groups` is a list of (bits, n,
    layer_offsets); width 1 runs the scaled-sign 1-bit Adam
    (OneBitOptimizer), the others a CodecGroup configured with `seed` (the
    library keys each width's uniforms by seed + bits).  Steps run the
    groups in list order."""

    def __init__(self, groups, W, chunk=1 << 20, align=4096, grad_dtype="f32", device="cuda",
                 period=10, seed=1234, sign_momentum=False, reset_interval=0, **hp):
        self.groups = []
        for bits, n, off in groups:
            if bits == 1:
                g = OneBitOptimizer(n, W, chunk, align, grad_dtype, off, device=device,
                                    sign_momentum=sign_momentum,
                                    reset_interval=reset_interval, **hp)
            else:
                g = CodecGroup(n, W, bits, align, grad_dtype, device, period, seed,
                               reset_interval, **hp)
            self.groups.append((bits, g))

    def close(self):
        for _, g in self.groups:
            g.close()

    def grad_buffers(self):
        return [g.grad_buffers() for _, g in self.groups]

    def warmup_step(self, grads, stream=None):
        for (_, g), gr in zip(self.groups, grads):
            g.warmup_step(gr, stream)

    def begin_compression(self, stream=None):
        for _, g in self.groups:
            g.begin_compression(stream)

    def compressed_step(self, grads, stream=None):
        for (_, g), gr in zip(self.groups, grads):
            g.compressed_step(gr, stream)
