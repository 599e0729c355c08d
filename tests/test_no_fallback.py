"""The product path has no CPU or library fallback: without libgdn.so the
binding raises, and host tensors are refused before any call is made."""
import pytest
import torch

from gated_deltanet_linear_02_gb300 import inputs as I
from gated_deltanet_linear_02_gb300 import ops


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(ops, "LIB_PATH", str(tmp_path / "libgdn.so"))
    monkeypatch.setattr(ops, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        ops.lib()


def test_host_tensors_are_refused():
    lp = I.layer_params(I.seed_of(0))
    st = I.streams(I.seed_of(0), 1, torch.bfloat16, lead=(2,))
    conv, S = I.initial_states(I.seed_of(0), 2, torch.bfloat16)
    out = torch.empty(2, I.D_INNER, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops.decode_step(lp, st.qkv[:, 0], st.z[:, 0], st.alpha[:, 0], st.beta[:, 0], conv, S, out)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ops.out_proj(torch.zeros(4, I.D_INNER, dtype=torch.bfloat16),
                     torch.zeros(I.N_EMBD, I.D_INNER, dtype=torch.bfloat16),
                     torch.zeros(4, I.N_EMBD, dtype=torch.bfloat16))
