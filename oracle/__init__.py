"""fp64 CPU oracle (test infrastructure only; see psk_oracle's header)."""
from .psk_oracle import *  # noqa: F401,F403
from .psk_oracle import (to_f64, exact_to_storage, page_summaries, summary_after_append, quest_scores, quest_scores_per_query_head,
                         forced_pages, select_pages, cutoff_score, retained_count, budget_for, page_masses, group_masses,
                         select_coverage, page_mean_std, gaussian_scores, latent_values, softmax_attention, page_tokens,
                         attend_pages, attend_pages_per_query_head, dense_attention, logical_from_cache, decode_step, default_scale)
