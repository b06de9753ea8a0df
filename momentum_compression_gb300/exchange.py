"""One rank of a multi-process 1-bit job over torch.distributed: one worker
and one server per process, the 3-phase compressed exchange of the 1-bit
LAMB summary (paragraphs 2 and 4) -- local compression, an all-to-all of
the compressed chunks, each server's average and re-compression, an
all-gather of the result -- with every computation in libob's kernels
(ob_compress_worker, ob_server_reduce_part, ob_adam_step / ob_lamb_step)
and only the two collectives here.

Block layout (the ctx's layout, W = the number of ranks, P the partition
size, cpp its chunks): a rank's compressed row holds partition i's words at
[i*P/32, (i+1)*P/32) and its scales at [i*cpp, (i+1)*cpp), so the
all-to-all sends these blocks as they are; rank j receives recv_bits
[W][P/32] and recv_scales [W][cpp] (row w from rank w), reduces partition
j, and the all-gather of the W partitions' outputs in rank order is the
whole server output.  The backend is the process group's: NCCL for device
tensors on a GPU job, gloo for host tensors.
"""
import momentum_compression_gb300 as ob


def _dist():
    import torch.distributed as dist
    return dist


def block_sizes(layout):
    """(words, scales) per block: P/32 sign words and cpp chunk scales."""
    return layout["P"] // 32, layout["chunks_per_partition"]


def exchange_worker_blocks(bits_row, scales_row, layout, recv_bits, recv_scales, group=None):
    """The all-to-all: block i of this rank's row (int32 words, float32
    scales) goes to rank i; recv_bits [W][P/32] and recv_scales [W][cpp]
    receive row w from rank w."""
    dist = _dist()
    W = layout["W"]
    wp, cpp = block_sizes(layout)
    dist.all_to_all_single(recv_bits.view(-1), bits_row.view(-1)[: W * wp], group=group)
    dist.all_to_all_single(recv_scales.view(-1), scales_row.view(-1)[: W * cpp], group=group)


def gather_server(sbits_part, sscales_part, layout, sbits, sscales, group=None):
    """The all-gather: the W partitions' server words and scales, in rank
    order, into the whole sbits (its first n_pad/32 words) and sscales."""
    dist = _dist()
    W = layout["W"]
    wp, cpp = block_sizes(layout)
    dist.all_gather_into_tensor(sbits.view(-1)[: W * wp], sbits_part.view(-1), group=group)
    dist.all_gather_into_tensor(sscales.view(-1), sscales_part.view(-1), group=group)


class RankOptimizer:
    """The buffers and call order of one rank: its own gradient and error,
    its row of compressed words and scales, the received blocks, its
    partition's server error and output, and the replicated m, v, p (and
    v_fresh, LAMB state) that every rank updates identically from the
    gathered server output.  With sign_momentum the momentum is held in its
    sign form (the gathered output) after the first compressed step; for
    1-bit LAMB the gathered output is then double-buffered, since the update
    reads the previous step's words too (server_targets names the pair this
    step's all-gather fills)."""

    def __init__(self, n, world, rank, chunk, align=4096, grad_dtype="f32",
                 layer_offsets=None, lamb=False, sign_momentum=False, group=None,
                 device="cuda", reset_interval=0, **hp):
        """reset_interval > 0: the periodic error reset, before the steps the
        library's plan names (ob_plan_step), as in OneBitOptimizer."""
        import torch
        self.rank, self.world, self.group, self.lamb = rank, world, group, lamb
        self.sign_momentum, self.m_in_signs = sign_momentum, False
        self.double_buffered = bool(sign_momentum and lamb)
        self.reset_interval, self.cstep = reset_interval, 0
        self.ctx = ob.ob_init(n, world, chunk, align,
                              ob.OB_GRAD_BF16 if grad_dtype == "bf16" else ob.OB_GRAD_F32,
                              layer_offsets, reset_interval=reset_interval, **hp)
        lay = ob.ob_get_layout(self.ctx)
        self.layout = lay
        wp, cpp = block_sizes(lay)
        z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=device)
        self.n_pad = lay["n_pad"]
        self.m, self.v, self.p = z(self.n_pad), z(self.n_pad), z(self.n_pad)
        self.v_fresh = z(self.n_pad) if lamb else None
        self.err = z(self.n_pad)
        self.bits_row = z(lay["words_per_worker"], dt=torch.int32)
        self.scales_row = z(lay["n_chunks"])
        self.recv_bits = z(world, wp, dt=torch.int32)
        self.recv_scales = z(world, cpp)
        self.err_s_part = z(lay["P"])
        self.sbits_part = z(wp, dt=torch.int32)
        self.sscales_part = z(cpp)
        self.sbits = z(lay["words_per_worker"], dt=torch.int32)
        self.sscales = z(lay["n_chunks"])
        self.sbits_alt = z(lay["words_per_worker"], dt=torch.int32) if self.double_buffered else None
        self.sscales_alt = z(lay["n_chunks"]) if self.double_buffered else None
        nbytes = ob.ob_workspace_bytes(self.ctx)
        self.workspace = z((nbytes + 255) // 256 * 64)
        ob.ob_set_workspace(self.ctx, self.workspace, nbytes)
        self.ls = ob.LayerState(lay["n_layers"], device) if lamb else None
        self.warmup_steps = 0

    def close(self):
        if self.ctx:
            ob.ob_destroy(self.ctx)
            self.ctx = None

    def warmup_step(self, grads_all):
        """An uncompressed step from all W gradients (gathered in rank order)."""
        ob.ob_warmup_step(self.ctx, grads_all, self.m, self.v, self.p,
                          ob.OB_MODE_LAMB if self.lamb else ob.OB_MODE_ADAM, self.ls)
        self.warmup_steps += 1

    def begin_compression(self):
        for t in (self.err, self.bits_row, self.scales_row, self.err_s_part, self.sbits_part,
                  self.sscales_part, self.sbits, self.sscales, self.sbits_alt, self.sscales_alt):
            if t is not None:
                t.zero_()
        self.cstep = 0
        if self.lamb:
            ob.ob_begin_compression(self.ctx, None, None, None, None, None, None, self.m,
                                    self.v, self.v_fresh, self.ls, max(self.warmup_steps, 1))
        self.m_in_signs = False

    def begin_step(self):
        """Counts the compressed step and, when the plan says so, resets this
        rank's worker error and its server partition's error first."""
        self.cstep += 1
        if self.reset_interval and ob.ob_plan_step(self.ctx, 1, self.cstep)["reset"]:
            ob.ob_reset_errors_rank(self.ctx, self.rank, self.err, self.bits_row,
                                    self.scales_row, self.err_s_part, self.sbits_part,
                                    self.sscales_part)

    def compress(self, grad):
        if self.m_in_signs:
            # m_{t-1} = sscale*sign (over sigma_l for LAMB) from the last gathered output
            ob.ob_compress_worker(self.ctx, grad, self.err, self.bits_row, self.scales_row,
                                  msbits=self.sbits, msscales=self.sscales, ls=self.ls)
        else:
            ob.ob_compress_worker(self.ctx, grad, self.err, self.bits_row, self.scales_row,
                                  m=self.m, ls=self.ls)

    def server(self):
        # in place: each tile's previous words and scale are read before it
        # is rewritten, and only the gathered copies feed the update
        ob.ob_server_reduce_part(self.ctx, self.rank, self.recv_bits, self.recv_scales,
                                 self.err_s_part, self.sbits_part, self.sscales_part, self.ls)

    def server_targets(self):
        """The whole-output buffers this step's all-gather fills: the current
        pair, or -- 1-bit LAMB in sign form after its first compressed step --
        the other pair, so that the update still sees the previous words."""
        if self.double_buffered and self.m_in_signs:
            return self.sbits_alt, self.sscales_alt
        return self.sbits, self.sscales

    def update(self):
        if self.double_buffered and self.m_in_signs:
            ob.ob_lamb_step_signm(self.ctx, self.sbits, self.sscales, self.sbits_alt,
                                  self.sscales_alt, self.v, self.v_fresh, self.p, self.ls)
            self.sbits, self.sbits_alt = self.sbits_alt, self.sbits
            self.sscales, self.sscales_alt = self.sscales_alt, self.sscales
        elif self.lamb:
            ob.ob_lamb_step(self.ctx, self.sbits, self.sscales, self.v, self.v_fresh, self.m,
                            self.p, self.ls)
            self.m_in_signs = self.sign_momentum
        else:
            ob.ob_adam_step(self.ctx, self.sbits, self.sscales, self.v,
                            None if self.sign_momentum else self.m, self.p)
            self.m_in_signs = self.sign_momentum

    def compressed_step(self, grad):
        """One compressed step of this rank; every rank of the group calls it
        together."""
        self.begin_step()
        self.compress(grad)
        exchange_worker_blocks(self.bits_row, self.scales_row, self.layout, self.recv_bits,
                               self.recv_scales, self.group)
        self.server()
        sbits, sscales = self.server_targets()
        gather_server(self.sbits_part, self.sscales_part, self.layout, sbits, sscales,
                      self.group)
        self.update()
