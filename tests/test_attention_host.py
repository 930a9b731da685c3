"""gna_attention's argument checks, which run on the host before any call into
the library (CPU tensors suffice: nothing reaches the device)."""
import pytest
import torch

from dimensional_sparse_attention_gna_b300 import gna_attention


def test_gna_attention_refuses_bad_inputs_on_host():
    x = torch.zeros((1, 1, 16, 16, 2, 32), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="bfloat16"):
        gna_attention(x.float(), x, x, (1, 5, 5))
    with pytest.raises(ValueError, match="one shape"):
        gna_attention(x, x[..., :16], x, (1, 5, 5))
    with pytest.raises(ValueError, match="one shape"):
        gna_attention(x[0], x[0], x[0], (1, 5, 5))
