"""libspecverify: target-side speculative-decoding verification on one GB300.

The compute path is the C-ABI library ``libspecverify.so`` (hand-written
CUDA for sm_103a, built in-tree by ``build.py``); ``api`` binds its calls for
torch tensors, ``step`` drives a whole verification step, ``workloads``
draws the seeded synthetic inputs.
"""

from .api import (Batch, BlockPool, PagedKV, sv_accept, sv_accept_workspace, sv_chunk_windows,
                  sv_commit_kv, sv_select_budget, sv_select_budget_workspace, sv_tree_attend,
                  sv_tree_attend_workspace, sv_verify_chunked, sv_verify_chunked_workspace,
                  workspace)
from ._native import SpecVerifyError

__all__ = ["Batch", "BlockPool", "PagedKV", "SpecVerifyError", "sv_accept", "sv_accept_workspace",
           "sv_chunk_windows", "sv_commit_kv", "sv_select_budget", "sv_select_budget_workspace",
           "sv_tree_attend", "sv_tree_attend_workspace", "sv_verify_chunked",
           "sv_verify_chunked_workspace", "workspace"]
