"""Paged grouped-query attention decode step for GB300 (sm_103a)."""
