"""One POET-X transformed linear held on the GPU, driven through the C ABI.

``TransformedLinear`` owns the device buffers of one layer (merged weight,
permutations and their inverses, skew parameters, the Cayley-Neumann blocks,
the saved activation and the workspace) and calls the C entry points in the
order of one training step:

  1. poetx_cayley_neumann_pair (P and R)  [POET-X §2.C-§2.D]
  2. poetx_forward   y = R (W0 (P x))      [POET-X §2.A-§2.C]
  3. poetx_backward  dX, dtheta_P, dtheta_R

and, when an inner loop ends, ``merge_and_resample`` (poetx_fold_w0, then
fresh permutations merged by poetx_merge_w0) [POET-X §2.B].  With
``w0_int8`` the merged weight is kept as INT8 codes and per-row scales
(POET-XQ, §2.E) and the _xq entry points dequantise it per call.

(source: "POET-X: Memory-efficient LLM Training by Scaling Orthogonal
Transformation", gist.science summary, section 2).  PyTorch only allocates
the buffers and supplies the stream; every step runs in the library's kernels.
``capture_step`` records one step's launches into a CUDA graph, so that a
training loop pays one host launch per step instead of one per kernel.
"""
import torch

from . import _lib


class TransformedLinear:
    def __init__(self, W0, theta_P, theta_R, perm_in, perm_out, b_in, b_out, n, T_max,
                 save_z=True, device="cuda", w0_int8=False, workspace=None):
        dev = torch.device(device)
        self.dtype = W0.dtype
        self.d_out, self.d_in = W0.shape
        self.b_in, self.b_out, self.n = int(b_in), int(b_out), int(n)
        self.T_max = int(T_max)
        self.save_z = save_z
        self.W0 = W0.to(dev).contiguous()
        self.theta_P = theta_P.to(dev, torch.float32).contiguous()
        self.theta_R = theta_R.to(dev, torch.float32).contiguous()
        self.perm_in = perm_in.to(dev, torch.int32).contiguous()
        self.perm_out = perm_out.to(dev, torch.int32).contiguous()
        self.inv_in = torch.empty_like(self.perm_in)
        self.inv_out = torch.empty_like(self.perm_out)
        _lib.poetx_invert_perm(self.perm_in, self.inv_in)
        _lib.poetx_invert_perm(self.perm_out, self.inv_out)
        # [§2.B] merge the two inner permutations into W0 once (per inner loop)
        self.W0m = torch.empty_like(self.W0)
        _lib.poetx_merge_w0(self.W0, self.W0m, self.perm_out, self.perm_in)
        # [§2.E] POET-XQ: keep only INT8 codes and per-row scales of the merged
        # weight resident; every forward / backward dequantises them into its
        # workspace
        self.w0_int8 = bool(w0_int8)
        self.W0q = self.w0_scale = None
        if self.w0_int8:
            self.W0q = torch.empty(self.d_out, self.d_in, dtype=torch.int8, device=dev)
            self.w0_scale = torch.empty(self.d_out, dtype=torch.float32, device=dev)
            _lib.poetx_quantize_w0(self.W0m, self.W0q, self.w0_scale)
            self.W0 = self.W0m = None
        nbi, nbo = self.d_in // self.b_in, self.d_out // self.b_out
        self.Q_P = torch.empty(nbi, self.b_in, self.b_in, dtype=self.dtype, device=dev)
        self.Q_R = torch.empty(nbo, self.b_out, self.b_out, dtype=self.dtype, device=dev)
        self.dtheta_P = torch.empty_like(self.theta_P)
        self.dtheta_R = torch.empty_like(self.theta_R)
        ws_bytes = (_lib.poetx_workspace_bytes_xq if self.w0_int8 else _lib.poetx_workspace_bytes)
        ws = ws_bytes(self.T_max, self.d_in, self.d_out, self.b_in, self.b_out, self.dtype)
        if ws == 0:
            raise ValueError("invalid layer sizes")
        # layers that run one after another on one stream may share one
        # workspace (the scratch of a call is dead once the call's kernels end)
        if workspace is not None:
            if workspace.dtype != torch.uint8 or workspace.numel() < ws:
                raise ValueError("shared workspace too small: need %d bytes" % ws)
            self.workspace = workspace
        else:
            self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.z = (torch.empty(self.T_max, self.d_out, dtype=self.dtype, device=dev)
                  if save_z else None)

    def cayley_neumann(self):
        _lib.poetx_cayley_neumann_pair(self.theta_P, self.b_in, self.theta_R, self.b_out, self.n,
                                       self.Q_P, self.Q_R)

    def forward(self, x, y=None):
        T = x.shape[0]
        if y is None:
            y = torch.empty(T, self.d_out, dtype=self.dtype, device=x.device)
        z = self.z[:T] if self.z is not None else None
        if self.w0_int8:
            _lib.poetx_forward_xq(x, self.W0q, self.w0_scale, self.Q_P, self.Q_R, self.perm_in,
                                  self.inv_in, self.perm_out, self.inv_out, self.b_in, self.b_out,
                                  y, z, self.workspace)
        else:
            _lib.poetx_forward(x, self.W0m, self.Q_P, self.Q_R, self.perm_in, self.inv_in,
                               self.perm_out, self.inv_out, self.b_in, self.b_out, y, z,
                               self.workspace)
        return y

    def backward(self, x, dy, dX=None):
        T = x.shape[0]
        if dX is None:
            dX = torch.empty(T, self.d_in, dtype=self.dtype, device=x.device)
        z = self.z[:T] if self.z is not None else None
        if self.w0_int8:
            _lib.poetx_backward_xq(x, dy, self.W0q, self.w0_scale, self.theta_P, self.theta_R,
                                   self.n, self.Q_P, self.Q_R, z, self.perm_in, self.inv_in,
                                   self.perm_out, self.inv_out, self.b_in, self.b_out, dX,
                                   self.dtheta_P, self.dtheta_R, self.workspace)
        else:
            _lib.poetx_backward(x, dy, self.W0m, self.theta_P, self.theta_R, self.n, self.Q_P,
                                self.Q_R, z, self.perm_in, self.inv_in, self.perm_out,
                                self.inv_out, self.b_in, self.b_out, dX, self.dtheta_P,
                                self.dtheta_R, self.workspace)
        return dX, self.dtheta_P, self.dtheta_R

    def step(self, x, dy, y=None, dX=None):
        """One pass of the whole hot path: CNP of both sides, forward, backward."""
        self.cayley_neumann()
        y = self.forward(x, y)
        dX, dtp, dtr = self.backward(x, dy, dX)
        return y, dX, dtp, dtr

    def merge_and_resample(self, perm_in, perm_out):
        """End of an inner loop [§2.B]: fold the current rotations into the
        frozen weight (W0 <- R W0 P, poetx_fold_w0), reset theta to zero (so
        Q = I), take the new permutations and merge them into the weight
        (poetx_merge_w0).  The layer then computes the same function as
        before, up to the fold's rounding, with fresh permutations."""
        self.cayley_neumann()                       # Q of the current theta
        dev = self.Q_P.device
        need = _lib.poetx_fold_workspace_bytes(self.d_out, self.d_in, self.b_in, self.b_out,
                                               self.dtype)
        if need == 0:
            raise ValueError("invalid layer sizes")
        ws = (self.workspace if self.workspace.numel() >= need else
              torch.empty(need, dtype=torch.uint8, device=dev))
        if self.w0_int8:   # the bf16 weights exist only while the fold runs
            W0m = torch.empty(self.d_out, self.d_in, dtype=self.dtype, device=dev)
            _lib.poetx_dequantize_w0(self.W0q, self.w0_scale, W0m)
            W0 = torch.empty_like(W0m)
        else:
            W0m, W0 = self.W0m, self.W0
        _lib.poetx_fold_w0(W0m, self.Q_P, self.Q_R, self.perm_in, self.perm_out, self.b_in,
                           self.b_out, W0, ws)
        self.theta_P.zero_()
        self.theta_R.zero_()
        self.perm_in.copy_(perm_in.to(torch.int32))
        self.perm_out.copy_(perm_out.to(torch.int32))
        _lib.poetx_invert_perm(self.perm_in, self.inv_in)
        _lib.poetx_invert_perm(self.perm_out, self.inv_out)
        _lib.poetx_merge_w0(W0, W0m, self.perm_out, self.perm_in)
        if self.w0_int8:
            _lib.poetx_quantize_w0(W0m, self.W0q, self.w0_scale)
        self.cayley_neumann()

    def capture_step(self, x, dy, y, dX, warm=True):
        """Capture one step on fixed buffers into a CUDA graph and return it.

        ``graph.replay()`` re-runs the whole step (the same kernels with the
        same arguments) on whatever ``x``, ``dy`` and the parameters hold at
        replay time, writing ``y``, ``dX`` and the skew gradients.  With
        ``warm`` the step first runs once eagerly on a side stream, so every
        launch's one-time set-up is done before capture."""
        if warm:
            side = torch.cuda.Stream(device=x.device)
            side.wait_stream(torch.cuda.current_stream(x.device))
            with torch.cuda.stream(side):
                self.step(x, dy, y, dX)
            torch.cuda.current_stream(x.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="relaxed"):
            self.step(x, dy, y, dX)
        return graph
