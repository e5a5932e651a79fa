"""One engine step's decode-attention calls captured once as a CUDA graph.

The SimpleLLM engine captures "CUDA graphs for any set of active slots, all
captured at startup" (README, changes table). Here one graph is enough for
every set of active slots: the kernels read the lengths and block tables on
the device (an inactive slot has length 0) and split the work there, so no
launch parameter depends on which slots are active or how long they are.
Change seq_lens, block tables and inputs in place, then replay().
"""
import torch

from . import decode_attn_reserve, decode_attn_workspace_bytes

__all__ = ["DecodeStepGraph"]


class DecodeStepGraph:
    """Capture `calls` (argument-free callables, each one library call on static
    buffers, in step order) into a single CUDA graph.

    shape = (batch, num_q_heads, num_kv_heads, head_dim) sizes the library
    workspace, which is reserved before capture (nothing is allocated inside it).
    """

    def __init__(self, calls, shape, device=None):
        self.calls = list(calls)
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.graph = None
        self.stream = None
        self.shape = shape

    def capture(self):
        with torch.cuda.device(self.device):
            decode_attn_reserve(decode_attn_workspace_bytes(*self.shape))
            self.stream = torch.cuda.Stream()
            self.stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(self.stream):  # warm-up: module load, kernel attributes
                for call in self.calls:
                    call()
            self.stream.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(self.graph, stream=self.stream):
                    for call in self.calls:
                        call()
            torch.cuda.current_stream().wait_stream(self.stream)
        return self

    def replay(self):
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
