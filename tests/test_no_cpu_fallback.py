"""The binding has no CPU path: every call refuses host tensors before it reaches the
library (which itself only launches CUDA kernels), and a missing library is an error,
not a silent fallback."""
import os

import pytest
import torch

import tree_speculative_decoding_verify_gb300 as T
from tree_speculative_decoding_verify_gb300 import _lib


def cpu(*shape, dtype=torch.int32):
    return torch.zeros(*shape, dtype=dtype)


CALLS = [
    ("lm_head_argmax", lambda: T.lm_head_argmax(cpu(4, 64, dtype=torch.bfloat16),
                                                cpu(10, 64, dtype=torch.bfloat16), cpu(4),
                                                cpu(256, dtype=torch.uint8))),
    ("tree_build_meta", lambda: T.tree_build_meta(cpu(1, 8), cpu(1), cpu(1), 3, cpu(1, 8, 1),
                                                  cpu(1, 8), cpu(1, 8, 4), cpu(1), cpu(1, 8),
                                                  cpu(1, 8))),
    ("accept_and_compact", lambda: T.accept_and_compact(cpu(1, 8), cpu(1, 8), cpu(1, 8),
                                                        cpu(1, 8), cpu(1), cpu(1), 3, None,
                                                        cpu(1, 4), cpu(1), cpu(1), cpu(1, 4, 2),
                                                        cpu(1))),
    ("draft_to_target", lambda: T.draft_to_target(cpu(1, 8), cpu(1), cpu(10))),
    ("draft_grow_mask", lambda: T.draft_grow_mask(cpu(1, 8, 1), cpu(1, 8), cpu(1, 2), cpu(1), 1)),
    ("target_probs", lambda: T.target_probs(cpu(1, 8, 10, dtype=torch.float32),
                                            cpu(1, dtype=torch.float32), cpu(1),
                                            cpu(1, dtype=torch.float32),
                                            cpu(1, dtype=torch.float32), cpu(1),
                                            cpu(1, 8, 10, dtype=torch.float32),
                                            cpu(256, dtype=torch.uint8))),
    ("draft_fixed_level", lambda: T.draft_fixed_level(cpu(1, 1, 10, dtype=torch.float32), 2, 1,
                                                      0, cpu(1, 8), cpu(1, 8))),
]


@pytest.mark.parametrize("name,call", CALLS, ids=[c[0] for c in CALLS])
def test_host_tensors_are_refused(name, call):
    with pytest.raises((TypeError, ValueError), match="CUDA"):
        call()


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", os.path.join(str(tmp_path), "libtsv.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(_lib.TsvError):
        _lib.lib()
